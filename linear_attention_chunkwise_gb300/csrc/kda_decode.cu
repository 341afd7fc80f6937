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
#include "kda_ptx.cuh"

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

// Both decode kernels reduce in the same order, so that a multi-token launch is bitwise equal to
// single steps: k . q by one warp (lane l takes channels 4l..4l+3 in an fma chain, then a butterfly
// over the lanes), and the column sums over the 8 groups of 16 rows as the pairwise tree
// ((g0 + g1) + (g2 + g3)) + ((g4 + g5) + (g6 + g7)).
__device__ __forceinline__ float warp_dot4(float4 x, float4 y) {
    float d = x.x * y.x;
    d = fmaf(x.y, y.y, d);
    d = fmaf(x.z, y.z, d);
    d = fmaf(x.w, y.w, d);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    return d;
}
__device__ __forceinline__ float warp_dot128(const float* a, const float* b, int lane) {
    return warp_dot4(reinterpret_cast<const float4*>(a)[lane], reinterpret_cast<const float4*>(b)[lane]);
}
// Four consecutive outputs from floats (8- or 16-byte aligned).
__device__ __forceinline__ void st4o(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4o(__nv_bfloat16* p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 r;
    r.x = *reinterpret_cast<const uint32_t*>(&a);
    r.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = r;
}
// Four consecutive elements as floats (8- or 16-byte aligned).
__device__ __forceinline__ float4 ld4f(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4f(const __nv_bfloat16* p) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u), __uint_as_float(r.y << 16),
                       __uint_as_float(r.y & 0xffff0000u));
}
__device__ __forceinline__ float tree8(float g0, float g1, float g2, float g3, float g4, float g5, float g6,
                                       float g7) {
    return ((g0 + g1) + (g2 + g3)) + ((g4 + g5) + (g6 + g7));
}

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

    __shared__ float a_s[kHeadDim];
    __shared__ __align__(16) float k_s[kHeadDim];
    __shared__ __align__(16) float q_s[kHeadDim];
    __shared__ __align__(16) float u_s[kHeadDim];
    __shared__ __align__(16) float red_y[kThreads / 32][kHeadDim];
    __shared__ __align__(16) float red_p[kThreads / 32][kHeadDim];
    __shared__ float kq_s;
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
    if (warp == 0) {  // k . q of the raw rows
        const float kq = warp_dot128(k_s, q_s, lane);
        if (lane == 0) kq_s = kq;
    }
    __syncthreads();

    if (tid < kHeadDim) {
        const float yy = tree8(red_y[0][tid], red_y[1][tid], red_y[2][tid], red_y[3][tid], red_y[4][tid],
                               red_y[5][tid], red_y[6][tid], red_y[7][tid]);
        const float pp = tree8(red_p[0][tid], red_p[1][tid], red_p[2][tid], red_p[3][tid], red_p[4][tid],
                               red_p[5][tid], red_p[6][tid], red_p[7][tid]);
        float b = beta[tok];
        if (FUSED && (fz.flags & KDA_FUSE_BETA_SIGMOID)) b = 1.f / (1.f + expf(-b));
        const float u = b * (to_f32(v[tok * kHeadDim + tid]) - yy);
        const float kq = kq_s * (ik * iq);
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
// tokens, so it is read once and written once per launch.  Per token the
// arithmetic is the single-step kernel's factorised update.
//
// Layout: warp w owns columns 16w..16w+15 of the state for all 128 rows; lane
// (g = lane / 4, c = lane % 4) holds rows 16g..16g+15 of columns 16w+4c..+3
// (one float4 per row; a warp reads eight 64-byte row pieces per load).  The
// column sums y = S'^T k and p = S'^T q are then reductions over the 8 lane
// groups of a warp (three shuffle levels), every lane of a column quad ends
// with the full sums, computes u and o for its 4 columns itself, and applies
// S += k u^T to its own rows: a token needs no block barrier (one with the
// fused output gate, whose RMSNorm sums o^2 over all 8 warps).  The L2 norms
// and k.q of a batch of NB tokens are taken once, before its tokens.
//
// The grid is persistent (two CTAs per SM, each walking the (sequence, head)
// units with a stride of the grid).  While a CTA runs the tokens of one unit,
// the NEXT unit's 64 KB state (eight bulk copies, one per warp) and the q, k,
// v, log alpha (and gate) rows of its first NB tokens (16-byte cp.async pieces
// spread over all threads: a thread that issues a bulk copy is held ~0.1 us,
// so one per row would stall the chain) come into shared memory, and the SM's
// share of HBM stays busy through the token chain.  Tokens past the first NB
// of a unit are read with plain loads when their batch starts.  Measured at
// 256 x 32 units, bf16: T = 4 in 186 us (the state blocks packed without
// padding, so a quarter-warp's two row groups read the same banks: 198 us;
// 16-byte cp.async pieces for the state: 202-207 us; a CTA per unit with
// two block barriers per token: 253 us).
template <typename IoT>
struct MultiLayout {
    static constexpr int NB = sizeof(IoT) == 2 ? 8 : 4;           // tokens per batch (two CTAs per SM fit)
    static constexpr uint32_t ROW = kHeadDim * sizeof(IoT);         // one token's q / k / v / gate row
    // f32 [8 blocks][16 rows][128], block b (one bulk copy) at b * BLK floats: 16 floats of padding
    // per block put the row groups a quarter-warp reads (16 rows apart) in different banks
    static constexpr uint32_t BLK = 16 * kHeadDim + 16;
    static constexpr uint32_t STATE = 0;
    static constexpr uint32_t Q = 8 * BLK * 4;                      // IoT [NB][128] each
    static constexpr uint32_t K = Q + NB * ROW;
    static constexpr uint32_t V = K + NB * ROW;
    static constexpr uint32_t G = V + NB * ROW;
    static constexpr uint32_t LA = G + NB * ROW;                    // f32 [NB][128]
    static constexpr uint32_t BAR = LA + NB * kHeadDim * 4;
    static constexpr uint32_t TOTAL = BAR + 16;
};

// Sums a float4 with the same float4 of lane (lane ^ off): a butterfly step.
__device__ __forceinline__ float4 shfl_xor4(float4 v, int off) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
    v.z += __shfl_xor_sync(0xffffffffu, v.z, off);
    v.w += __shfl_xor_sync(0xffffffffu, v.w, off);
    return v;
}

// FUSED: the prologue / epilogue of DecodeFusion, per token (as kda_decode_kernel's).
template <typename IoT, bool FUSED>
__global__ void __launch_bounds__(kThreads, 2)
    kda_decode_multi_kernel(const IoT* __restrict__ q, const IoT* __restrict__ k, const IoT* __restrict__ v,
                            const float* __restrict__ log_alpha, const float* __restrict__ beta, float* S,
                            int32_t num_slots, const int32_t* __restrict__ state_indices, int32_t T, int32_t H,
                            int32_t units, IoT* __restrict__ o, float* S_steps, int32_t* device_status,
                            const DecodeFusion fz) {
    using L = MultiLayout<IoT>;
    constexpr int NB = L::NB;
    extern __shared__ __align__(128) uint8_t dsm[];
    float* const st_buf = reinterpret_cast<float*>(dsm + L::STATE);
    uint64_t* const bar = reinterpret_cast<uint64_t*>(dsm + L::BAR);

    __shared__ __align__(16) float a_s[NB][kHeadDim];
    __shared__ __align__(16) float k_s[NB][kHeadDim];
    __shared__ __align__(16) float q_s[NB][kHeadDim];
    __shared__ __align__(16) float v_s[NB][kHeadDim];
    __shared__ __align__(16) float g_s[FUSED ? NB : 1][FUSED ? kHeadDim : 4];  // output gates of the batch
    __shared__ float b_s[NB], kq_s[NB];
    __shared__ float b_raw[NB];          // the fetched unit's beta (or logits) of its first nb0 tokens
    __shared__ float oo_part[2][kThreads / 32];  // o^2 per warp, by token parity (output gate)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool l2n = FUSED && (fz.flags & KDA_FUSE_L2NORM_QK);
    const bool og = FUSED && (fz.flags & KDA_FUSE_OUT_GATE);
    const bool sig = FUSED && (fz.flags & KDA_FUSE_BETA_SIGMOID);
    const int nb0 = min(NB, T);
    const int r0 = 16 * (lane >> 2);              // this lane's first row
    const int c0 = 16 * warp + 4 * (lane & 3);    // this lane's first column

    auto slot_of = [&](int u) { return state_indices ? state_indices[u / H] : u / H; };
    // Unit u's 64 KB state (when `slot` is valid) as eight 8 KB bulk copies, one issued by lane 0 of each
    // warp (a thread that issues a bulk copy is held for a while, so no warp issues more than one); thread
    // 0 posts the byte count on the barrier first (post_state, before the CTA barrier that precedes
    // fetch_state; a bare arrival when the slot is out of range).
    auto post_state = [&](int32_t slot) {
        if (tid == 0) mbar_arrive_expect_tx(bar, (slot >= 0 && slot < num_slots) ? kHeadDim * kHeadDim * 4u : 0u);
    };
    auto fetch_state = [&](int u, int32_t slot) {
        if (slot >= 0 && slot < num_slots && lane == 0)
            bulk_g2s(st_buf + warp * L::BLK,
                     S + ((static_cast<size_t>(slot) * H + (u % H)) * kHeadDim + 16 * warp) * kHeadDim,
                     16 * kHeadDim * 4u, bar);
    };
    // Every thread: 16-byte pieces of the q, k, v, log alpha (and gate) rows of unit u's first nb0 tokens,
    // and (tid < nb0) token tid's beta, by cp.async without a register stage; each thread waits for its
    // own pieces (cp.async.wait_all) before the barrier that precedes their first use.
    auto fetch_inputs = [&](int u) {
        constexpr int CR = L::ROW / 16;                // pieces per q / k / v / gate row
        const int per_tok = (og ? 4 : 3) * CR + 32;    // + 32 pieces of log alpha
        const int n = u / H, h = u - n * H;
        for (int e = tid; e < nb0 * per_tok; e += kThreads) {
            const int tt = e / per_tok, r = e - tt * per_tok;
            const size_t row = ((static_cast<size_t>(n) * T + tt) * H + h) * kHeadDim;
            const void* src;
            uint32_t dst;
            if (r < 32) {
                src = log_alpha + row + 4 * r;
                dst = L::LA + tt * 512u + 16u * r;
            } else {
                const int a = (r - 32) / CR, c = (r - 32) - a * CR;
                const IoT* base = a == 0 ? q : a == 1 ? k : a == 2 ? v : static_cast<const IoT*>(fz.out_gate);
                src = reinterpret_cast<const uint8_t*>(base + row) + 16 * c;
                dst = (a == 0 ? L::Q : a == 1 ? L::K : a == 2 ? L::V : L::G) + tt * L::ROW + 16u * c;
            }
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dsm + dst)),
                         "l"(reinterpret_cast<uint64_t>(src))
                         : "memory");
        }
        if (tid < nb0) {
            const float* src = beta + (static_cast<size_t>(n) * T + tid) * H + h;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(&b_raw[tid])),
                         "l"(reinterpret_cast<uint64_t>(src))
                         : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // Warp tt: token tt of the batch, lane l taking channels 4l..4l+3: its k, q, v, log alpha (and gate)
    // rows to fp32 (from the fetched rows, or from global at row `tok`), alpha = exp(log alpha), the L2
    // norms of k and q (prologue), k . q and beta.
    auto convert_token = [&](int tt, bool fetched, size_t tok) {
        float4 k4, q4, v4, l4, g4 = make_float4(0.f, 0.f, 0.f, 0.f);
        float bb;
        if (fetched) {
            const int off = tt * kHeadDim + 4 * lane;
            k4 = ld4f(reinterpret_cast<const IoT*>(dsm + L::K) + off);
            q4 = ld4f(reinterpret_cast<const IoT*>(dsm + L::Q) + off);
            v4 = ld4f(reinterpret_cast<const IoT*>(dsm + L::V) + off);
            l4 = ld4f(reinterpret_cast<const float*>(dsm + L::LA) + off);
            if (og) g4 = ld4f(reinterpret_cast<const IoT*>(dsm + L::G) + off);
            bb = b_raw[tt];
        } else {
            const size_t off = tok * kHeadDim + 4 * lane;
            k4 = ld4f(k + off);
            q4 = ld4f(q + off);
            v4 = ld4f(v + off);
            l4 = ld4f(log_alpha + off);
            if (og) g4 = ld4f(static_cast<const IoT*>(fz.out_gate) + off);
            bb = beta[tok];
        }
        if (l2n) {
            float k2 = k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w;
            float q2 = q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w;
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) {
                k2 += __shfl_xor_sync(0xffffffffu, k2, o2);
                q2 += __shfl_xor_sync(0xffffffffu, q2, o2);
            }
            const float ik = rsqrtf(k2 + fz.l2_eps), iq = rsqrtf(q2 + fz.l2_eps);
            k4.x *= ik; k4.y *= ik; k4.z *= ik; k4.w *= ik;
            q4.x *= iq; q4.y *= iq; q4.z *= iq; q4.w *= iq;
        }
        const float kq = warp_dot4(k4, q4);
        reinterpret_cast<float4*>(k_s[tt])[lane] = k4;
        reinterpret_cast<float4*>(q_s[tt])[lane] = q4;
        reinterpret_cast<float4*>(v_s[tt])[lane] = v4;
        reinterpret_cast<float4*>(a_s[tt])[lane] = make_float4(expf(l4.x), expf(l4.y), expf(l4.z), expf(l4.w));
        if (og) reinterpret_cast<float4*>(g_s[tt])[lane] = g4;
        if (lane == 0) {
            kq_s[tt] = kq;
            b_s[tt] = sig ? 1.f / (1.f + expf(-bb)) : bb;
        }
    };

    int u = blockIdx.x;
    int32_t slot = u < units ? slot_of(u) : 0;
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        if (u < units) post_state(slot);
    }
    __syncthreads();
    if (u < units) {
        fetch_state(u, slot);
        fetch_inputs(u);
    }

    for (uint32_t phase = 0; u < units; u += gridDim.x, phase ^= 1u) {
        const int n = u / H, h = u - n * H;
        const int32_t cur = slot;
        const bool valid = cur >= 0 && cur < num_slots;
        const int un = u + static_cast<int>(gridDim.x);
        const int32_t nslot = un < units ? slot_of(un) : 0;  // the next unit's slot, read early
        // every thread is past the previous unit's tokens, and this unit's copies have landed
        asm volatile("cp.async.wait_all;" ::: "memory");
        const bool late = !mbar_wait_pipe(bar, phase);
        if (__syncthreads_or(late)) {  // the copy waited for has drained: nothing is left in flight
            if (tid == 0 && device_status) atomicOr(device_status, KDA_DEV_TIMEOUT);
            return;
        }
        float4 s[16];
        if (valid) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                s[i] = *reinterpret_cast<const float4*>(st_buf + (lane >> 2) * L::BLK + i * kHeadDim + c0);
        }
        if (warp < nb0) convert_token(warp, true, 0);
        if (un < units) post_state(nslot);
        __syncthreads();  // the state and the fetched rows are consumed: fetch the next unit into them
        if (un < units) {
            fetch_state(un, nslot);
            fetch_inputs(un);
        }
        slot = nslot;
        if (!valid) {
            if (tid == 0 && device_status) atomicOr(device_status, KDA_DEV_BAD_SLOT);
            continue;
        }
        float* const Sg = S + (static_cast<size_t>(cur) * H + h) * kHeadDim * kHeadDim;

        for (int tb0 = 0; tb0 < T; tb0 += NB) {
            const int nb = min(NB, T - tb0);
            if (tb0 > 0) {
                __syncthreads();  // the previous batch's vectors are no longer read
                if (warp < nb) convert_token(warp, false, (static_cast<size_t>(n) * T + tb0 + warp) * H + h);
                __syncthreads();
            }

            for (int tt = 0; tt < nb; ++tt) {
                const size_t tok = (static_cast<size_t>(n) * T + tb0 + tt) * H + h;
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f), p = y;
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const float4 a4 = reinterpret_cast<const float4*>(a_s[tt] + r0)[i4];
                    const float4 k4 = reinterpret_cast<const float4*>(k_s[tt] + r0)[i4];
                    const float4 q4 = reinterpret_cast<const float4*>(q_s[tt] + r0)[i4];
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w},
                                qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float4& t = s[4 * i4 + j];
                        t.x *= av[j]; t.y *= av[j]; t.z *= av[j]; t.w *= av[j];
                        y.x = fmaf(kv[j], t.x, y.x); y.y = fmaf(kv[j], t.y, y.y);
                        y.z = fmaf(kv[j], t.z, y.z); y.w = fmaf(kv[j], t.w, y.w);
                        p.x = fmaf(qv[j], t.x, p.x); p.y = fmaf(qv[j], t.y, p.y);
                        p.z = fmaf(qv[j], t.z, p.z); p.w = fmaf(qv[j], t.w, p.w);
                    }
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {  // over the 8 row groups: full column sums
                    y = shfl_xor4(y, off);
                    p = shfl_xor4(p, off);
                }
                const float4 v4 = *reinterpret_cast<const float4*>(&v_s[tt][c0]);
                const float b = b_s[tt], kq = kq_s[tt];
                float4 uu, ov;
                uu.x = b * (v4.x - y.x); uu.y = b * (v4.y - y.y); uu.z = b * (v4.z - y.z); uu.w = b * (v4.w - y.w);
                ov.x = fmaf(kq, uu.x, p.x); ov.y = fmaf(kq, uu.y, p.y);
                ov.z = fmaf(kq, uu.z, p.z); ov.w = fmaf(kq, uu.w, p.w);
                if (og) {  // y = RMSNorm(o) * weight * gate: o^2 summed over the warp's 16 columns, then warps
                    float o2 = ov.x * ov.x + ov.y * ov.y + ov.z * ov.z + ov.w * ov.w;
                    o2 += __shfl_xor_sync(0xffffffffu, o2, 1);
                    o2 += __shfl_xor_sync(0xffffffffu, o2, 2);
                    if (lane == 0) oo_part[tt & 1][warp] = o2;
                    __syncthreads();  // a parity's partials are rewritten only after the next token's barrier
                    float ms = 0.f;
#pragma unroll
                    for (int w = 0; w < kThreads / 32; ++w) ms += oo_part[tt & 1][w];
                    const float rn = rsqrtf(ms * (1.f / kHeadDim) + fz.rms_eps);
                    const float4 g4 = *reinterpret_cast<const float4*>(&g_s[tt][c0]);
                    const float4 w4 = fz.rms_weight ? make_float4(fz.rms_weight[c0], fz.rms_weight[c0 + 1],
                                                                  fz.rms_weight[c0 + 2], fz.rms_weight[c0 + 3])
                                                    : make_float4(1.f, 1.f, 1.f, 1.f);
                    ov.x *= rn * w4.x * g4.x; ov.y *= rn * w4.y * g4.y;
                    ov.z *= rn * w4.z * g4.z; ov.w *= rn * w4.w * g4.w;
                }
                if (lane < 4) st4o(o + tok * kHeadDim + c0, ov);  // row group 0: the warp's 16 outputs
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const float4 k4 = reinterpret_cast<const float4*>(k_s[tt] + r0)[i4];
                    const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float4& t = s[4 * i4 + j];
                        t.x = fmaf(kv[j], uu.x, t.x); t.y = fmaf(kv[j], uu.y, t.y);
                        t.z = fmaf(kv[j], uu.z, t.z); t.w = fmaf(kv[j], uu.w, t.w);
                    }
                }
                if (S_steps) {
                    float* const Ss = S_steps + tok * kHeadDim * kHeadDim;
#pragma unroll
                    for (int i = 0; i < 16; ++i) __stcs(reinterpret_cast<float4*>(Ss + (r0 + i) * kHeadDim + c0), s[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) __stcs(reinterpret_cast<float4*>(Sg + (r0 + i) * kHeadDim + c0), s[i]);
    }
}

}  // namespace

// Persistent grid of the multi-token kernel: as many CTAs as fit on the device at once (two per SM),
// never more than there are units.  The occupancy is looked up once per device and instantiation.
template <typename IoT, bool FUSED>
cudaError_t launch_multi_t(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                           float* S, int32_t num_slots, const int32_t* state_indices, int32_t T, int32_t H,
                           int32_t units, void* o, float* S_steps, int32_t* device_status, cudaStream_t stream,
                           const DecodeFusion& fz) {
    constexpr uint32_t smem = MultiLayout<IoT>::TOTAL;
    static int resident[64];  // CTAs that fit on the device at once, per device (0: not looked up yet)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    int fit = (dev >= 0 && dev < 64) ? resident[dev] : 0;
    if (fit == 0) {
        err = cudaFuncSetAttribute(kda_decode_multi_kernel<IoT, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        int sms = 0, per_sm = 0;
        err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_decode_multi_kernel<IoT, FUSED>, kThreads,
                                                            smem);
        if (err != cudaSuccess) return err;
        fit = sms * (per_sm > 0 ? per_sm : 1);
        if (dev >= 0 && dev < 64) resident[dev] = fit;
    }
    const dim3 grid(static_cast<unsigned>(units < fit ? units : fit));
    kda_decode_multi_kernel<IoT, FUSED><<<grid, kThreads, smem, stream>>>(
        static_cast<const IoT*>(q), static_cast<const IoT*>(k), static_cast<const IoT*>(v), log_alpha, beta, S,
        num_slots, state_indices, T, H, units, static_cast<IoT*>(o), S_steps, device_status, fz);
    return cudaGetLastError();
}

cudaError_t launch_decode_multi(bool f32_io, const void* q, const void* k, const void* v, const float* log_alpha,
                                const float* beta, float* S, int32_t num_slots, const int32_t* state_indices,
                                int32_t N, int32_t T, int32_t H, void* o, float* S_steps, int32_t* device_status,
                                cudaStream_t stream, const DecodeFusion& fusion) {
    const long long units = static_cast<long long>(N) * H;
    if (units == 0 || T == 0) return cudaSuccess;
    if (T == 1 && !S_steps)  // one token: the single-step kernel (the same arithmetic, no staging)
        return launch_decode(f32_io, q, k, v, log_alpha, beta, S, num_slots, state_indices, N, H, o, device_status,
                             stream, fusion);
    const int32_t nu = static_cast<int32_t>(units);
    const bool fused = fusion.flags != 0;
    if (f32_io)
        return (fused ? launch_multi_t<float, true> : launch_multi_t<float, false>)(
            q, k, v, log_alpha, beta, S, num_slots, state_indices, T, H, nu, o, S_steps, device_status, stream,
            fusion);
    return (fused ? launch_multi_t<__nv_bfloat16, true> : launch_multi_t<__nv_bfloat16, false>)(
        q, k, v, log_alpha, beta, S, num_slots, state_indices, T, H, nu, o, S_steps, device_status, stream, fusion);
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
