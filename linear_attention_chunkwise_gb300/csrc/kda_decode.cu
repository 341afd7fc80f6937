// kda_decode.cu -- fused single-token KDA update ("fused recurrent mode").
//
// One CTA per (sequence, head).  The head's 128 x 128 fp32 state is streamed
// through registers exactly once: 256 threads, thread (warp w, lane l) holds
// rows 16w..16w+15, columns 4l..4l+3 (one float4 per row, so every warp reads
// and writes whole 512-byte rows).  The update is evaluated in the factorised
// form that needs a single pass over the state:
//   S' = Diag(alpha) S                         (rows = key channels)
//   y  = S'^T k,  p = S'^T q                   (column sums over the 128 rows)
//   u  = beta (v - y)
//   S_new = S' + k u^T                         (= (I - beta k k^T) S' + beta k v^T)
//   o  = S_new^T q = p + (k . q) u
// which is the KDA equation of "Understanding Kimi Delta Attention"
// (pyshine), "The KDA Recurrence: Scalar Gate vs Channel-wise Gate",
// rewritten with the erase-then-write delta form of "kimi delta attn from
// first principles" (aryagxr), section "KDA", step 2.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = kHeadDim / (kThreads / 32);  // 16

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// FUSED adds the prologue / epilogue of DecodeFusion: q, k L2-normalised,
// beta = sigmoid(logit), output y = RMSNorm(o) * weight * gate (the three
// gates of "kimi delta attn from first principles" (aryagxr), "KDA has three
// gates", and its "KDA Architecture" L2 norm).
template <typename IoT, bool FUSED>
__global__ void __launch_bounds__(kThreads, 2)
    kda_decode_kernel(const IoT* __restrict__ q, const IoT* __restrict__ k, const IoT* __restrict__ v,
                      const float* __restrict__ log_alpha, const float* __restrict__ beta, float* S,
                      int32_t num_slots, const int32_t* __restrict__ state_indices, int32_t H,
                      IoT* __restrict__ o, int32_t* device_status, const DecodeFusion fz) {
    const int unit = blockIdx.x;
    const int n = unit / H;
    const int h = unit - n * H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int32_t slot = state_indices ? state_indices[n] : n;
    if (slot < 0 || slot >= num_slots) {
        if (tid == 0 && device_status) atomicOr(device_status, KDA_DEV_BAD_SLOT);
        return;
    }

    __shared__ float a_s[kHeadDim], k_s[kHeadDim], q_s[kHeadDim];
    __shared__ __align__(16) float u_s[kHeadDim];
    __shared__ __align__(16) float red_y[kThreads / 32][kHeadDim];
    __shared__ __align__(16) float red_p[kThreads / 32][kHeadDim];
    __shared__ float kq_part[4];
    __shared__ float kk_part[4], qq_part[4], oo_part[4];

    float* Sg = S + (static_cast<size_t>(slot) * H + h) * kHeadDim * kHeadDim;
    const int row0 = warp * kRowsPerWarp;

    // Issue the whole 64 KB state read up front (16 independent float4 per thread).
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        s[i] = __ldcs(reinterpret_cast<const float4*>(Sg + static_cast<size_t>(row0 + i) * kHeadDim) + lane);

    const size_t tok = static_cast<size_t>(n) * H + h;
    if (tid < kHeadDim) {
        const float kk = to_f32(k[tok * kHeadDim + tid]);
        const float qq = to_f32(q[tok * kHeadDim + tid]);
        k_s[tid] = kk;
        q_s[tid] = qq;
        a_s[tid] = expf(log_alpha[tok * kHeadDim + tid]);
        float kq = kk * qq;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (lane == 0) kq_part[warp] = kq;
        if (FUSED && (fz.flags & KDA_FUSE_L2NORM_QK)) {
            float k2 = kk * kk, q2 = qq * qq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                k2 += __shfl_xor_sync(0xffffffffu, k2, off);
                q2 += __shfl_xor_sync(0xffffffffu, q2, off);
            }
            if (lane == 0) { kk_part[warp] = k2; qq_part[warp] = q2; }
        }
    }
    __syncthreads();
    // L2 norms of k and q (1 without the prologue); the rows below use k/|k|, q/|q|
    float ik = 1.f, iq = 1.f;
    if (FUSED && (fz.flags & KDA_FUSE_L2NORM_QK)) {
        ik = rsqrtf(kk_part[0] + kk_part[1] + kk_part[2] + kk_part[3] + fz.l2_eps);
        iq = rsqrtf(qq_part[0] + qq_part[1] + qq_part[2] + qq_part[3] + fz.l2_eps);
    }

    float o_val = 0.f;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f), p = y;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = row0 + i;
        const float a = a_s[r], kr = k_s[r] * ik, qr = q_s[r] * iq;
        s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
        y.x = fmaf(kr, s[i].x, y.x); y.y = fmaf(kr, s[i].y, y.y);
        y.z = fmaf(kr, s[i].z, y.z); y.w = fmaf(kr, s[i].w, y.w);
        p.x = fmaf(qr, s[i].x, p.x); p.y = fmaf(qr, s[i].y, p.y);
        p.z = fmaf(qr, s[i].z, p.z); p.w = fmaf(qr, s[i].w, p.w);
    }
    reinterpret_cast<float4*>(red_y[warp])[lane] = y;
    reinterpret_cast<float4*>(red_p[warp])[lane] = p;
    __syncthreads();

    if (tid < kHeadDim) {
        float yy = 0.f, pp = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            yy += red_y[w][tid];
            pp += red_p[w][tid];
        }
        float b = beta[tok];
        if (FUSED && (fz.flags & KDA_FUSE_BETA_SIGMOID)) b = 1.f / (1.f + expf(-b));
        const float u = b * (to_f32(v[tok * kHeadDim + tid]) - yy);
        const float kq = (kq_part[0] + kq_part[1] + kq_part[2] + kq_part[3]) * (ik * iq);
        u_s[tid] = u;
        o_val = fmaf(kq, u, pp);
        if (FUSED && (fz.flags & KDA_FUSE_OUT_GATE)) {
            float o2 = o_val * o_val;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) o2 += __shfl_xor_sync(0xffffffffu, o2, off);
            if (lane == 0) oo_part[warp] = o2;
        } else {
            o[tok * kHeadDim + tid] = from_f32<IoT>(o_val);
        }
    }
    __syncthreads();
    if (FUSED && (fz.flags & KDA_FUSE_OUT_GATE) && tid < kHeadDim) {  // y = RMSNorm(o) * weight * gate
        const float ms = (oo_part[0] + oo_part[1] + oo_part[2] + oo_part[3]) * (1.f / kHeadDim);
        const float w = fz.rms_weight ? fz.rms_weight[tid] : 1.f;
        const float g = to_f32(static_cast<const IoT*>(fz.out_gate)[tok * kHeadDim + tid]);
        o[tok * kHeadDim + tid] = from_f32<IoT>(o_val * rsqrtf(ms + fz.rms_eps) * w * g);
    }

    const float4 uu = reinterpret_cast<const float4*>(u_s)[lane];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const float kr = k_s[row0 + i] * ik;
        float4 t = s[i];
        t.x = fmaf(kr, uu.x, t.x); t.y = fmaf(kr, uu.y, t.y);
        t.z = fmaf(kr, uu.z, t.z); t.w = fmaf(kr, uu.w, t.w);
        __stcs(reinterpret_cast<float4*>(Sg + static_cast<size_t>(row0 + i) * kHeadDim) + lane, t);
    }
}

// T consecutive tokens per sequence in one launch (a speculative-decoding
// verify step, or a short prefill): the state stays in registers across the
// tokens, so it is read once and written once per launch.  The per-token
// arithmetic is the single-step kernel's, token after token.  The inputs of up
// to kTokBatch tokens are fetched into shared memory up front (together with
// the state read), so no token waits on a global load: each token costs two
// block barriers (column partial sums, then u).
constexpr int kTokBatch = 8;

// FUSED: the prologue / epilogue of DecodeFusion, per token (as kda_decode_kernel's).
template <typename IoT, bool FUSED>
__global__ void __launch_bounds__(kThreads, 2)
    kda_decode_multi_kernel(const IoT* __restrict__ q, const IoT* __restrict__ k, const IoT* __restrict__ v,
                            const float* __restrict__ log_alpha, const float* __restrict__ beta, float* S,
                            int32_t num_slots, const int32_t* __restrict__ state_indices, int32_t T, int32_t H,
                            IoT* __restrict__ o, float* S_steps, int32_t* device_status, const DecodeFusion fz) {
    const int unit = blockIdx.x;
    const int n = unit / H;
    const int h = unit - n * H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int32_t slot = state_indices ? state_indices[n] : n;
    if (slot < 0 || slot >= num_slots) {
        if (tid == 0 && device_status) atomicOr(device_status, KDA_DEV_BAD_SLOT);
        return;
    }

    __shared__ float a_s[kTokBatch][kHeadDim], k_s[kTokBatch][kHeadDim], q_s[kTokBatch][kHeadDim];
    __shared__ float v_s[kTokBatch][kHeadDim], b_s[kTokBatch];
    __shared__ __align__(16) float u_s[kHeadDim];
    __shared__ __align__(16) float red_y[kThreads / 32][kHeadDim];
    __shared__ __align__(16) float red_p[kThreads / 32][kHeadDim];
    __shared__ float kq_part[4];
    __shared__ float g_s[FUSED ? kTokBatch : 1][FUSED ? kHeadDim : 1];  // output gates of the batch
    __shared__ float oo_part[4];
    const bool l2n = FUSED && (fz.flags & KDA_FUSE_L2NORM_QK);
    const bool og = FUSED && (fz.flags & KDA_FUSE_OUT_GATE);

    float* Sg = S + (static_cast<size_t>(slot) * H + h) * kHeadDim * kHeadDim;
    const int row0 = warp * kRowsPerWarp;
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        s[i] = __ldcs(reinterpret_cast<const float4*>(Sg + static_cast<size_t>(row0 + i) * kHeadDim) + lane);

    for (int tb0 = 0; tb0 < T; tb0 += kTokBatch) {
        const int nb = min(kTokBatch, T - tb0);
        if (tb0 > 0) __syncthreads();  // the previous batch's vectors are no longer read
        for (int e = tid; e < nb * kHeadDim; e += kThreads) {
            const int tt = e / kHeadDim, ch = e - tt * kHeadDim;
            const size_t tok = (static_cast<size_t>(n) * T + tb0 + tt) * H + h;
            k_s[tt][ch] = to_f32(k[tok * kHeadDim + ch]);
            q_s[tt][ch] = to_f32(q[tok * kHeadDim + ch]);
            a_s[tt][ch] = expf(log_alpha[tok * kHeadDim + ch]);
            v_s[tt][ch] = to_f32(v[tok * kHeadDim + ch]);
            if (og) g_s[tt][ch] = to_f32(static_cast<const IoT*>(fz.out_gate)[tok * kHeadDim + ch]);
        }
        if (tid < nb) {
            float bb = beta[(static_cast<size_t>(n) * T + tb0 + tid) * H + h];
            if (FUSED && (fz.flags & KDA_FUSE_BETA_SIGMOID)) bb = 1.f / (1.f + expf(-bb));
            b_s[tid] = bb;
        }
        __syncthreads();
        if (l2n) {  // warp tt normalises token tt's k and q rows in place
            if (warp < nb) {
                float k2 = 0.f, q2 = 0.f;
#pragma unroll
                for (int c = lane; c < kHeadDim; c += 32) {
                    k2 = fmaf(k_s[warp][c], k_s[warp][c], k2);
                    q2 = fmaf(q_s[warp][c], q_s[warp][c], q2);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    k2 += __shfl_xor_sync(0xffffffffu, k2, off);
                    q2 += __shfl_xor_sync(0xffffffffu, q2, off);
                }
                const float ik = rsqrtf(k2 + fz.l2_eps), iq = rsqrtf(q2 + fz.l2_eps);
#pragma unroll
                for (int c = lane; c < kHeadDim; c += 32) {
                    k_s[warp][c] *= ik;
                    q_s[warp][c] *= iq;
                }
            }
            __syncthreads();
        }

        for (int tt = 0; tt < nb; ++tt) {
            float o_val = 0.f;
            const int t = tb0 + tt;
            const size_t tok = (static_cast<size_t>(n) * T + t) * H + h;
            float4 y = make_float4(0.f, 0.f, 0.f, 0.f), p = y;
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const int r = row0 + i;
                const float a = a_s[tt][r], kr = k_s[tt][r], qr = q_s[tt][r];
                s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
                y.x = fmaf(kr, s[i].x, y.x); y.y = fmaf(kr, s[i].y, y.y);
                y.z = fmaf(kr, s[i].z, y.z); y.w = fmaf(kr, s[i].w, y.w);
                p.x = fmaf(qr, s[i].x, p.x); p.y = fmaf(qr, s[i].y, p.y);
                p.z = fmaf(qr, s[i].z, p.z); p.w = fmaf(qr, s[i].w, p.w);
            }
            reinterpret_cast<float4*>(red_y[warp])[lane] = y;
            reinterpret_cast<float4*>(red_p[warp])[lane] = p;
            if (tid < kHeadDim) {
                float kq = k_s[tt][tid] * q_s[tt][tid];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
                if (lane == 0) kq_part[warp] = kq;
            }
            __syncthreads();

            if (tid < kHeadDim) {
                float yy = 0.f, pp = 0.f;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) {
                    yy += red_y[w][tid];
                    pp += red_p[w][tid];
                }
                const float u = b_s[tt] * (v_s[tt][tid] - yy);
                const float kq = kq_part[0] + kq_part[1] + kq_part[2] + kq_part[3];
                u_s[tid] = u;
                o_val = fmaf(kq, u, pp);
                if (og) {
                    float o2 = o_val * o_val;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) o2 += __shfl_xor_sync(0xffffffffu, o2, off);
                    if (lane == 0) oo_part[warp] = o2;
                } else {
                    o[tok * kHeadDim + tid] = from_f32<IoT>(o_val);
                }
            }
            __syncthreads();
            if (og && tid < kHeadDim) {  // y = RMSNorm(o) * weight * gate; oo_part is rewritten only after
                                         // the next token's first barrier
                const float ms = (oo_part[0] + oo_part[1] + oo_part[2] + oo_part[3]) * (1.f / kHeadDim);
                const float w = fz.rms_weight ? fz.rms_weight[tid] : 1.f;
                o[tok * kHeadDim + tid] = from_f32<IoT>(o_val * rsqrtf(ms + fz.rms_eps) * w * g_s[tt][tid]);
            }

            const float4 uu = reinterpret_cast<const float4*>(u_s)[lane];
            float* Ss = S_steps ? S_steps + tok * kHeadDim * kHeadDim : nullptr;
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const float kr = k_s[tt][row0 + i];
                s[i].x = fmaf(kr, uu.x, s[i].x); s[i].y = fmaf(kr, uu.y, s[i].y);
                s[i].z = fmaf(kr, uu.z, s[i].z); s[i].w = fmaf(kr, uu.w, s[i].w);
                if (Ss) __stcs(reinterpret_cast<float4*>(Ss + static_cast<size_t>(row0 + i) * kHeadDim) + lane, s[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        __stcs(reinterpret_cast<float4*>(Sg + static_cast<size_t>(row0 + i) * kHeadDim) + lane, s[i]);
}

}  // namespace

template <typename IoT, bool FUSED>
void launch_multi_t(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta, float* S,
                    int32_t num_slots, const int32_t* state_indices, int32_t T, int32_t H, void* o, float* S_steps,
                    int32_t* device_status, cudaStream_t stream, const DecodeFusion& fz, dim3 grid) {
    kda_decode_multi_kernel<IoT, FUSED><<<grid, kThreads, 0, stream>>>(
        static_cast<const IoT*>(q), static_cast<const IoT*>(k), static_cast<const IoT*>(v), log_alpha, beta, S,
        num_slots, state_indices, T, H, static_cast<IoT*>(o), S_steps, device_status, fz);
}

cudaError_t launch_decode_multi(bool f32_io, const void* q, const void* k, const void* v, const float* log_alpha,
                                const float* beta, float* S, int32_t num_slots, const int32_t* state_indices,
                                int32_t N, int32_t T, int32_t H, void* o, float* S_steps, int32_t* device_status,
                                cudaStream_t stream, const DecodeFusion& fusion) {
    const long long units = static_cast<long long>(N) * H;
    if (units == 0 || T == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(units));
    const bool fused = fusion.flags != 0;
    if (f32_io)
        (fused ? launch_multi_t<float, true> : launch_multi_t<float, false>)(
            q, k, v, log_alpha, beta, S, num_slots, state_indices, T, H, o, S_steps, device_status, stream, fusion,
            grid);
    else
        (fused ? launch_multi_t<__nv_bfloat16, true> : launch_multi_t<__nv_bfloat16, false>)(
            q, k, v, log_alpha, beta, S, num_slots, state_indices, T, H, o, S_steps, device_status, stream, fusion,
            grid);
    return cudaGetLastError();
}

template <typename IoT, bool FUSED>
void launch_decode_t(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                     float* S, int32_t num_slots, const int32_t* state_indices, int32_t H, void* o,
                     int32_t* device_status, cudaStream_t stream, const DecodeFusion& fz, dim3 grid) {
    kda_decode_kernel<IoT, FUSED><<<grid, kThreads, 0, stream>>>(
        static_cast<const IoT*>(q), static_cast<const IoT*>(k), static_cast<const IoT*>(v), log_alpha, beta, S,
        num_slots, state_indices, H, static_cast<IoT*>(o), device_status, fz);
}

cudaError_t launch_decode(bool f32_io, const void* q, const void* k, const void* v, const float* log_alpha,
                          const float* beta, float* S, int32_t num_slots, const int32_t* state_indices,
                          int32_t N, int32_t H, void* o, int32_t* device_status, cudaStream_t stream,
                          const DecodeFusion& fusion) {
    const long long units = static_cast<long long>(N) * H;
    if (units == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(units));
    const bool fused = fusion.flags != 0;
    if (f32_io) {
        (fused ? launch_decode_t<float, true> : launch_decode_t<float, false>)(
            q, k, v, log_alpha, beta, S, num_slots, state_indices, H, o, device_status, stream, fusion, grid);
    } else {
        (fused ? launch_decode_t<__nv_bfloat16, true> : launch_decode_t<__nv_bfloat16, false>)(
            q, k, v, log_alpha, beta, S, num_slots, state_indices, H, o, device_status, stream, fusion, grid);
    }
    return cudaGetLastError();
}

}  // namespace kda
