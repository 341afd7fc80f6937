// kda_backward.cu -- gradient of the KDA prefill (reverse mode, fp32).
//
// For a loss L = sum_t <o_t, dO_t> + sum_n <S_final_n, dS_final_n> the adjoint
// of the state is carried backward token by token through the update of
// "Understanding Kimi Delta Attention" (pyshine), "The KDA Recurrence", in the
// erase-then-write form of "kimi delta attn from first principles" (aryagxr),
// "KDA":
//   S' = Diag(a) S_{t-1},  r = v - S'^T k,  u = beta r,  S_t = S' + k u^T,
//   o_t = S_t^T q.
// Per token, with G the adjoint of S_t (dS_final, plus what later tokens sent):
//   G += q dO^T;  dq = S_t dO;  du = G^T k;  dv = beta du;  dbeta = <du, r>;
//   dy = -beta du;  dk = G u + S' dy;  dS' = G + k dy^T;
//   dlog_alpha_i = a_i sum_j dS'_ij S_{t-1,ij} = sum_j dS'_ij S'_ij;  G <- Diag(a) dS'.
// Every column of S and of G evolves on its own (r, u, du, dy are per column),
// so a CTA owns one (sequence, head, column slice) and only dq, dk, dlog_alpha
// and dbeta -- sums over columns -- are shared between the slices of a head.
// The CTA walks its sequence backward chunk by chunk (64 tokens).  The state at
// the chunk start comes from the chunkwise prefill (a snapshot after every
// chunk); inside the chunk the per-token states are recomputed in fp32 into a
// per-CTA scratch slab and consumed in reverse.  State and adjoint live in
// registers: warp w holds rows 16w .. 16w+15, lane l holds CPT adjacent columns.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kBT = 256;                       // threads per CTA
constexpr int kBWarps = kBT / 32;
constexpr int kBRows = kHeadDim / kBWarps;     // 16 rows per warp
constexpr int kBC = kChunk;                    // tokens per chunk (64)

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// CPT adjacent floats (16, 8 or 4 bytes, aligned)
template <int CPT>
__device__ __forceinline__ void ldv(const float* p, float (&x)[CPT]) {
    if constexpr (CPT == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else if constexpr (CPT == 2) {
        const float2 t = *reinterpret_cast<const float2*>(p);
        x[0] = t.x; x[1] = t.y;
    } else {
        x[0] = *p;
    }
}
template <int CPT>
__device__ __forceinline__ void stv(float* p, const float (&x)[CPT]) {
    if constexpr (CPT == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else if constexpr (CPT == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    } else {
        *p = x[0];
    }
}

// Row totals of this warp's 16 rows (x[i] = this lane's partial of row 16w + i),
// reduce-scattered over the lanes: lanes l and l^1 end with the total of row
// 16w + row_of_lane(l).  16 shuffles.
__device__ __forceinline__ float row_sums(float (&x)[kBRows], int lane) {
#pragma unroll
    for (int half = kBRows / 2, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float send = upper ? x[j] : x[j + half];
            const float keep = upper ? x[j + half] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 1);
}
__device__ __forceinline__ int row_of_lane(int lane) {
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

template <int CPT>
struct BwdSmem {  // fp32 copies of one chunk (channel index innermost)
    static constexpr int NC = 32 * CPT;  // columns of the slice
    float q[kBC][kHeadDim];
    float k[kBC][kHeadDim];
    float a[kBC][kHeadDim];    // exp(log_alpha)
    float dO[kBC][kHeadDim];
    float r[kBC][NC];          // v, overwritten by r = v - S'^T k in the forward recompute
    float b[kBC];
    float red[kBWarps][NC];
    float dy[NC];
    float part[kBWarps];
    int unit;
};

// Work item i (longest sequences first) -> (sequence, head, slice).
template <typename IoT, int CPT>
__global__ void __launch_bounds__(kBT, 1)
    kda_backward_kernel(const IoT* __restrict__ q, const IoT* __restrict__ k, const IoT* __restrict__ v,
                        const float* __restrict__ log_alpha, const float* __restrict__ beta,
                        const float* __restrict__ S0, const int32_t* __restrict__ cu_seqlens,
                        const int32_t* __restrict__ order, const int32_t* __restrict__ chunk_off,
                        const float* __restrict__ ckpt, const IoT* __restrict__ dO,
                        const float* __restrict__ dS_final, float* __restrict__ dq, float* __restrict__ dk,
                        float* __restrict__ dv, float* __restrict__ dla, float* __restrict__ dbeta,
                        float* __restrict__ dS0, float* __restrict__ scratch, int32_t* __restrict__ work,
                        int32_t N, int32_t H) {
    constexpr int NC = 32 * CPT;
    constexpr int SL = kHeadDim / NC;  // slices per head
    constexpr bool kAtomic = SL > 1;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BwdSmem<CPT>& sm = *reinterpret_cast<BwdSmem<CPT>*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = warp * kBRows, myrow = row0 + row_of_lane(lane);
    const int lc = lane * CPT;  // first column of this lane within the slice
    if (chunk_off[N + 1] == 0) return;  // malformed cu_seqlens: the chunk table flagged it
    float* slab = scratch + static_cast<size_t>(blockIdx.x) * kBC * kHeadDim * NC;
    const int units = N * H * SL;

    for (;;) {
        __syncthreads();  // the previous unit's shared data is no longer read
        if (tid == 0) sm.unit = atomicAdd(work, 1);
        __syncthreads();
        const int unit = sm.unit;
        if (unit >= units) break;
        const int n = order[unit / (H * SL)];
        const int h = (unit / SL) % H, sl = unit % SL;
        const int c0 = sl * NC;  // first column of the slice
        const int64_t t_begin = cu_seqlens[n], t_end = cu_seqlens[n + 1];
        const int nch = chunk_off[n + 1] - chunk_off[n];
        const size_t sidx = (static_cast<size_t>(n) * H + h) * kHeadDim * kHeadDim;
        float G[kBRows][CPT];  // adjoint of the state after the current token
#pragma unroll
        for (int i = 0; i < kBRows; ++i) {
            if (dS_final) {
                ldv<CPT>(dS_final + sidx + (row0 + i) * kHeadDim + c0 + lc, G[i]);
            } else {
#pragma unroll
                for (int c = 0; c < CPT; ++c) G[i][c] = 0.f;
            }
        }

        for (int ch = nch - 1; ch >= 0; --ch) {
            const int64_t tc = t_begin + static_cast<int64_t>(ch) * kBC;
            const int L = static_cast<int>(t_end - tc < kBC ? t_end - tc : kBC);
            __syncthreads();  // the previous chunk's vectors are no longer read
            for (int e = tid; e < L * kHeadDim; e += kBT) {
                const int i = e / kHeadDim, c = e - i * kHeadDim;
                const size_t x = (static_cast<size_t>(tc + i) * H + h) * kHeadDim + c;
                sm.q[i][c] = ld_f32(q + x);
                sm.k[i][c] = ld_f32(k + x);
                sm.a[i][c] = expf(log_alpha[x]);
                sm.dO[i][c] = ld_f32(dO + x);
            }
            for (int e = tid; e < L * NC; e += kBT) {
                const int i = e / NC, c = e - i * NC;
                sm.r[i][c] = ld_f32(v + (static_cast<size_t>(tc + i) * H + h) * kHeadDim + c0 + c);
            }
            if (tid < L) sm.b[tid] = beta[(tc + tid) * H + h];
            // state at the chunk start: S0 for the first chunk, else the snapshot after chunk ch-1
            const float* Sst =
                ch == 0 ? (S0 ? S0 + sidx : nullptr)
                        : ckpt + (static_cast<size_t>(chunk_off[n] + ch - 1) * H + h) * kHeadDim * kHeadDim;
            float S[kBRows][CPT];
#pragma unroll
            for (int i = 0; i < kBRows; ++i) {
                if (Sst) {
                    ldv<CPT>(Sst + (row0 + i) * kHeadDim + c0 + lc, S[i]);
                } else {
#pragma unroll
                    for (int c = 0; c < CPT; ++c) S[i][c] = 0.f;
                }
            }
            __syncthreads();

            // forward recompute: S_{t-1} of every token to the slab, r = v - S'^T k to shared memory
            for (int i = 0; i < L; ++i) {
                float* srow = slab + static_cast<size_t>(i) * kHeadDim * NC;
                float y[CPT];
#pragma unroll
                for (int c = 0; c < CPT; ++c) y[c] = 0.f;
#pragma unroll
                for (int j = 0; j < kBRows; ++j) {
                    const int rr = row0 + j;
                    stv<CPT>(srow + rr * NC + lc, S[j]);
                    const float a = sm.a[i][rr], kr = sm.k[i][rr];
#pragma unroll
                    for (int c = 0; c < CPT; ++c) {
                        S[j][c] *= a;
                        y[c] = fmaf(kr, S[j][c], y[c]);
                    }
                }
                stv<CPT>(&sm.red[warp][lc], y);
                __syncthreads();
                if (tid < NC) {
                    float yy = 0.f;
#pragma unroll
                    for (int w = 0; w < kBWarps; ++w) yy += sm.red[w][tid];
                    sm.r[i][tid] -= yy;
                }
                __syncthreads();
                const float bi = sm.b[i];
                float u[CPT];
                ldv<CPT>(&sm.r[i][lc], u);
#pragma unroll
                for (int c = 0; c < CPT; ++c) u[c] *= bi;
#pragma unroll
                for (int j = 0; j < kBRows; ++j) {
                    const float kr = sm.k[i][row0 + j];
#pragma unroll
                    for (int c = 0; c < CPT; ++c) S[j][c] = fmaf(kr, u[c], S[j][c]);
                }
            }

            // reverse over the chunk's tokens (each thread reads back only the slab entries it wrote)
            for (int i = L - 1; i >= 0; --i) {
                const size_t tok = static_cast<size_t>(tc + i) * H + h;
                const float* srow = slab + static_cast<size_t>(i) * kHeadDim * NC;
                const float bi = sm.b[i];
                float u[CPT], d4[CPT];
                ldv<CPT>(&sm.r[i][lc], u);
#pragma unroll
                for (int c = 0; c < CPT; ++c) u[c] *= bi;
                ldv<CPT>(&sm.dO[i][c0 + lc], d4);
                float Sd[kBRows][CPT];  // S' = Diag(a) S_{t-1}
                float px[kBRows];
#pragma unroll
                for (int j = 0; j < kBRows; ++j) {
                    const int rr = row0 + j;
                    const float a = sm.a[i][rr], kr = sm.k[i][rr], qr = sm.q[i][rr];
                    ldv<CPT>(srow + rr * NC + lc, Sd[j]);
                    float p = 0.f;
#pragma unroll
                    for (int c = 0; c < CPT; ++c) {
                        Sd[j][c] *= a;
                        p = fmaf(fmaf(kr, u[c], Sd[j][c]), d4[c], p);  // (S_t dO) partial
                        G[j][c] = fmaf(qr, d4[c], G[j][c]);            // G += q dO^T
                    }
                    px[j] = p;
                }
                const float dqr = row_sums(px, lane);
                // du = G^T k (column sums over the 128 rows)
                float du[CPT];
#pragma unroll
                for (int c = 0; c < CPT; ++c) du[c] = 0.f;
#pragma unroll
                for (int j = 0; j < kBRows; ++j) {
                    const float kr = sm.k[i][row0 + j];
#pragma unroll
                    for (int c = 0; c < CPT; ++c) du[c] = fmaf(kr, G[j][c], du[c]);
                }
                stv<CPT>(&sm.red[warp][lc], du);
                __syncthreads();
                if (tid < NC) {
                    float d = 0.f;
#pragma unroll
                    for (int w = 0; w < kBWarps; ++w) d += sm.red[w][tid];
                    dv[tok * kHeadDim + c0 + tid] = bi * d;
                    sm.dy[tid] = -bi * d;
                    float pb = d * sm.r[i][tid];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, off);
                    if (lane == 0) sm.part[warp] = pb;
                }
                __syncthreads();
                if (tid == 0) {
                    float db = 0.f;
#pragma unroll
                    for (int w = 0; w < NC / 32; ++w) db += sm.part[w];
                    if (kAtomic) atomicAdd(dbeta + tok, db);
                    else dbeta[tok] = db;
                }
                float dy[CPT];
                ldv<CPT>(&sm.dy[lc], dy);
                // dk = G u + S' dy;  dS' = G + k dy^T;  dla = rowsum(dS' o S');  G <- Diag(a) dS'
                float pk[kBRows], pa[kBRows];
#pragma unroll
                for (int j = 0; j < kBRows; ++j) {
                    const float kr = sm.k[i][row0 + j], a = sm.a[i][row0 + j];
                    float s1 = 0.f, s2 = 0.f;
#pragma unroll
                    for (int c = 0; c < CPT; ++c) {
                        s1 = fmaf(G[j][c], u[c], s1);
                        s1 = fmaf(Sd[j][c], dy[c], s1);
                        const float ds = fmaf(kr, dy[c], G[j][c]);
                        s2 = fmaf(ds, Sd[j][c], s2);
                        G[j][c] = a * ds;
                    }
                    pk[j] = s1;
                    pa[j] = s2;
                }
                const float dkr = row_sums(pk, lane);
                const float dar = row_sums(pa, lane);
                if ((lane & 1) == 0) {
                    const size_t o = tok * kHeadDim + myrow;
                    if (kAtomic) {
                        atomicAdd(dq + o, dqr);
                        atomicAdd(dk + o, dkr);
                        atomicAdd(dla + o, dar);
                    } else {
                        dq[o] = dqr;
                        dk[o] = dkr;
                        dla[o] = dar;
                    }
                }
            }
        }
        if (dS0) {
#pragma unroll
            for (int i = 0; i < kBRows; ++i) stv<CPT>(dS0 + sidx + (row0 + i) * kHeadDim + c0 + lc, G[i]);
        }
    }
}

// Snapshot entries for every chunk end of every sequence: entry chunk_off[n] + c - 1 is the state
// after chunk c - 1 of sequence n (c = 1 .. nch_n; the last is the final state).  Entries past the
// batch's chunk count are sentinels (sequence N) that no scan CTA takes.
__global__ void kda_ckpt_entries_kernel(const int32_t* __restrict__ cu_seqlens,
                                        const int32_t* __restrict__ chunk_off, int32_t N, int32_t max_entries,
                                        int32_t* __restrict__ snap_seq, int32_t* __restrict__ snap_pos) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n > N) return;
    const bool valid = chunk_off[N + 1] != 0;
    if (n == N) {
        for (int e = valid ? chunk_off[N] : 0; e < max_entries; ++e) {
            snap_seq[e] = N;
            snap_pos[e] = 1;
        }
        return;
    }
    if (!valid) return;
    const int len = cu_seqlens[n + 1] - cu_seqlens[n];
    const int base = chunk_off[n], nch = chunk_off[n + 1] - base;
    for (int c = 1; c <= nch; ++c) {
        snap_seq[base + c - 1] = n;
        snap_pos[base + c - 1] = min(c * kBC, len);
    }
}

template <typename IoT, int CPT>
cudaError_t launch_backward_t(const BackwardArgs& a, int32_t ctas, cudaStream_t stream) {
    const size_t smem = sizeof(BwdSmem<CPT>);
    auto kern = kda_backward_kernel<IoT, CPT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    kern<<<ctas, kBT, smem, stream>>>(static_cast<const IoT*>(a.q), static_cast<const IoT*>(a.k),
                                      static_cast<const IoT*>(a.v), a.log_alpha, a.beta, a.S0, a.cu_seqlens, a.order,
                                      a.chunk_off, a.ckpt, static_cast<const IoT*>(a.dO), a.dS_final, a.dq, a.dk,
                                      a.dv, a.dla, a.dbeta, a.dS0, a.scratch, a.work, a.num_seqs, a.H);
    return cudaGetLastError();
}

}  // namespace

size_t backward_slab_bytes(int cols) { return static_cast<size_t>(kBC) * kHeadDim * cols * 4; }

cudaError_t launch_ckpt_entries(const int32_t* cu_seqlens, const int32_t* chunk_off, int32_t N, int32_t max_entries,
                                int32_t* snap_seq, int32_t* snap_pos, cudaStream_t stream) {
    const int threads = 128, blocks = (N + 1 + threads - 1) / threads;
    kda_ckpt_entries_kernel<<<blocks, threads, 0, stream>>>(cu_seqlens, chunk_off, N, max_entries, snap_seq,
                                                            snap_pos);
    return cudaGetLastError();
}

cudaError_t launch_backward(const BackwardArgs& a, bool f32_io, int32_t cols, int32_t ctas, cudaStream_t stream) {
    if (ctas <= 0) return cudaSuccess;
    if (f32_io) {
        if (cols == 128) return launch_backward_t<float, 4>(a, ctas, stream);
        if (cols == 64) return launch_backward_t<float, 2>(a, ctas, stream);
        if (cols == 32) return launch_backward_t<float, 1>(a, ctas, stream);
    } else {
        if (cols == 128) return launch_backward_t<__nv_bfloat16, 4>(a, ctas, stream);
        if (cols == 64) return launch_backward_t<__nv_bfloat16, 2>(a, ctas, stream);
        if (cols == 32) return launch_backward_t<__nv_bfloat16, 1>(a, ctas, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kda
