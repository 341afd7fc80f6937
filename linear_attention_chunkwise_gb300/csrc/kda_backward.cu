// kda_backward.cu -- chunkwise gradient of the KDA prefill (fp32).
//
// The function differentiated is the recurrence of "Understanding Kimi Delta
// Attention" (pyshine), "The KDA Recurrence", read in the erase-then-write
// order of "kimi delta attn from first principles" (aryagxr), "KDA":
//   S'_t = Diag(a_t) S_{t-1},  y_t = S'_t^T k_t,  u_t = beta_t (v_t - y_t),
//   S_t = S'_t + k_t u_t^T,  o_t = S_t^T q_t,
// for L = sum <o_t, dO_t> + <S_final, dS_final>.  Inside a 64-token chunk,
// with the chunkwise operands of "The Chunkwise DPLR Algorithm" (g the
// inclusive cumulative log-decay, gm = g of row 31, gC = g of the last row,
// Kh = k e^{g-gm}, Qh = q e^{g-gm}, Kb = k e^{gm-g}, Lm = strict lower Kh Kb^T,
// Mm = lower Qh Kb^T incl. diagonal, Tb = (I + Diag(beta) Lm)^-1 Diag(beta)),
// the chunk-start state S (Sm = Diag(e^{gm}) S) and the adjoint X of the state
// after the chunk (Xc = Diag(e^{gC-gm}) X), the gradient is a set of dense
// products:
//   U  = Tb (V - Kh Sm),  R = V - Kh Sm - Lm U          (rows beta_t r_t and r_t)
//   dY = -Tb^T (Mm^T dO + Kb Xc)   (dL/dy_t),  dv = -dY
//   du = Mm^T dO + Lm^T dY + Kb Xc,  dbeta_t = <du_t, r_t>
//   dq = Eq (dO Sm^T + tril(dO U^T) Kb),                        Eq = e^{g-gm}
//   dk = Eb (triu(U dO^T) Qh + striu(U dY^T) Kh + U Xc^T)         Eb = e^{gm-g}
//      + Eq (dY Sm^T + stril(dY U^T) Kb)
//   dg = q dq + k (second part of dk - first part);  last row += rowsum(S_next X)
//   dlog_alpha = reverse cumulative sum of dg over the chunk's rows
// and X walks back over chunks as X <- Diag(e^{gC}) X + Diag(e^{gm}) (Qh^T dO + Kh^T dY),
// dS0 = X before the first chunk.
//
// Kernels (all 256 threads; products on fp32 shared tiles as tf32 mma.sync, fp32 accumulation):
//   prep      per (chunk, head): the X-independent pieces -> a per-chunk record
//   scan      per (sequence, head, 32 state columns): the walk of X; writes dv = -dY,
//             X after every chunk and its columns' part of rowsum(S_next X) (into the
//             consumed record)
//   value+key per (chunk, head): U, dbeta, then dq, dk, dlog_alpha (U, dO, dY kept in shared memory)
// The chunk-start states come from the chunkwise prefill (a snapshot after every chunk).
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_prefill_common.cuh"

namespace kda {
namespace {

constexpr int BT = 256;
constexpr int C = kChunk;     // 64
constexpr int D = kHeadDim;   // 128
constexpr int LDW = 132;      // row stride (floats) of 128-wide shared tiles: conflict-free column reads
constexpr int LDN = 68;       // of 64-wide tiles
constexpr int LDS = 36;       // of 32-wide tiles
constexpr int LDX = 40;       // of 32-wide tiles read as adjacent pairs in fragment layout (8 mod 32 words)
constexpr int TILE = C * LDW;
constexpr int PTILE = C * LDN;
constexpr int NCS = 32;       // state columns per scan CTA
constexpr int kSlices = D / NCS;
static_assert(kSlices == 4, "the boundary term sums four slice parts");

// per-(chunk, head) record of the prep kernel (fp32)
constexpr int kRecWbc = 0;        // [64][128]  Tb^T Kb Diag(e^{gC-gm})
constexpr int kRecDY0 = 8192;     // [64][128]  -Tb^T Mm^T dO
constexpr int kRecKhm = 16384;    // [64][128]  Kh Diag(e^{gm})
constexpr int kRecP = 24576;      // [128][128] Diag(e^{gm}) Qh^T dO
constexpr int kRecTb = 40960;     // [64][64]   Tb
constexpr int kRecGam = 45056;    // [128]      e^{gC}
constexpr int kRecFloats = 45184;

template <typename T>
__device__ __forceinline__ float4 ld4(const T* p);
template <>
__device__ __forceinline__ float4 ld4<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <typename T>
__device__ __forceinline__ void st4(T* p, float4 v);
template <>
__device__ __forceinline__ void st4<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <>
__device__ __forceinline__ void st4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = w;
}
// ---- products on shared tiles ---------------------------------------------------------------
// Tensor-core products of fp32 shared tiles: operands rounded to tf32 (cvt.rna), fp32 accumulate,
// mma.sync m16n8k8.  One warp owns 16 output rows from r0 and NT 8-column tiles from c0; its
// accumulator acc[j][e] holds row r0 + g + 8 (e >> 1), column c0 + 8 j + 2 t + (e & 1)
// (g = lane >> 2, t = lane & 3).  Operand element addressing:
//   AR: A(m, k) = A[m * lda + k]     AC: A(m, k) = A[k * lda + m]
//   BK: B(k, n) = B[k * ldb + n]     BN: B(k, n) = B[n * ldb + k]
//   BK8: as BK, for a B whose row stride is 8 mod 32 words (fragment k indices t, t + 4 conflict-free)
enum { AR = 0, AC = 1, BK = 0, BN = 1, BK8 = 2 };

// Inside a k-step the fragments may take the step's eight k indices in any order that A and B
// share.  With B(k, n) = B[k * ldb + n] (BK) lane (g, t) takes k = 2t, 2t + 1 instead of the
// fragment's t, t + 4: for the tiles' row strides (4 mod 32 words) the B reads then fall on 32
// distinct banks (t, t + 4 put two lanes on each of 16 banks), and so do the AC reads of A; the AR
// reads of A, a quarter of the loads, become two-way.
template <int NT, int AM, int BM>
__device__ __forceinline__ void mma16(float (&acc)[NT][4], const float* A, int lda, const float* B, int ldb, int K,
                                      int r0, int c0, int lane) {
    const int g = lane >> 2, t = lane & 3;
    if constexpr (BM == BK) {
#pragma unroll 2
        for (int k0 = 0; k0 < K; k0 += 8) {
            const int k = k0 + 2 * t;
            uint32_t a[4];
            if (AM == AR) {
                const float2 lo = *reinterpret_cast<const float2*>(A + (r0 + g) * lda + k);
                const float2 hi = *reinterpret_cast<const float2*>(A + (r0 + g + 8) * lda + k);
                a[0] = to_tf32(lo.x);
                a[1] = to_tf32(hi.x);
                a[2] = to_tf32(lo.y);
                a[3] = to_tf32(hi.y);
            } else {
                a[0] = to_tf32(A[k * lda + r0 + g]);
                a[1] = to_tf32(A[k * lda + r0 + g + 8]);
                a[2] = to_tf32(A[(k + 1) * lda + r0 + g]);
                a[3] = to_tf32(A[(k + 1) * lda + r0 + g + 8]);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int n = c0 + 8 * j + g;
                mma_tf32(acc[j], a, to_tf32(B[k * ldb + n]), to_tf32(B[(k + 1) * ldb + n]));
            }
        }
    } else {  // BN and BK8: the fragment's own k indices t, t + 4
#pragma unroll 2
        for (int k0 = 0; k0 < K; k0 += 8) {
            uint32_t a[4];
            if (AM == AR) {
                a[0] = to_tf32(A[(r0 + g) * lda + k0 + t]);
                a[1] = to_tf32(A[(r0 + g + 8) * lda + k0 + t]);
                a[2] = to_tf32(A[(r0 + g) * lda + k0 + t + 4]);
                a[3] = to_tf32(A[(r0 + g + 8) * lda + k0 + t + 4]);
            } else {
                a[0] = to_tf32(A[(k0 + t) * lda + r0 + g]);
                a[1] = to_tf32(A[(k0 + t) * lda + r0 + g + 8]);
                a[2] = to_tf32(A[(k0 + t + 4) * lda + r0 + g]);
                a[3] = to_tf32(A[(k0 + t + 4) * lda + r0 + g + 8]);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int n = c0 + 8 * j + g;
                if (BM == BN) mma_tf32(acc[j], a, to_tf32(B[n * ldb + k0 + t]), to_tf32(B[n * ldb + k0 + t + 4]));
                else mma_tf32(acc[j], a, to_tf32(B[(k0 + t) * ldb + n]), to_tf32(B[(k0 + t + 4) * ldb + n]));
            }
        }
    }
}
template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
}
// coordinates of accumulator element (j, e)
__device__ __forceinline__ int frow(int r0, int lane, int e) { return r0 + (lane >> 2) + 8 * (e >> 1); }
__device__ __forceinline__ int fcol(int c0, int lane, int j, int e) { return c0 + 8 * j + 2 * (lane & 3) + (e & 1); }

// ---- loads ------------------------------------------------------------------------------------
// rows [t0, t0 + L) of a [T, H, 128] tensor, head h -> fp32 tile (stride LDW), rows >= L zero.
// Constant trip counts: every thread's loads are in flight together.
template <typename T>
__device__ __forceinline__ void load_tile(float* dst, const T* src, int64_t t0, int L, int H, int h, int tid,
                                          float scale = 1.f) {
    constexpr int IT = C * (D / 4) / BT;  // 8
    float4 v[IT];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int e = tid + it * BT, r = e >> 5, c4 = (e & 31) * 4;
        v[it] = r < L ? ld4(src + (static_cast<size_t>(t0 + r) * H + h) * D + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int e = tid + it * BT, r = e >> 5, c4 = (e & 31) * 4;
        *reinterpret_cast<float4*>(dst + r * LDW + c4) =
            make_float4(v[it].x * scale, v[it].y * scale, v[it].z * scale, v[it].w * scale);
    }
}
__device__ __forceinline__ void cp16(float* dst, const float* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
// 16 bytes, or 16 zero bytes when !valid (nothing is read then; src must still be a mapped address)
__device__ __forceinline__ void cp16z(float* dst, const float* src, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Two such tiles with all sixteen loads of a thread in flight before its first store (separate
// calls would wait for the first tile's loads before issuing the second's).
template <typename TA, typename TB>
__device__ __forceinline__ void load_tile2(float* dst_a, const TA* src_a, float* dst_b, const TB* src_b, int64_t t0,
                                           int L, int H, int h, int tid, float scale_b = 1.f) {
    constexpr int IT = C * (D / 4) / BT;  // 8
    float4 va[IT], vb[IT];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int e = tid + it * BT, r = e >> 5, c4 = (e & 31) * 4;
        const size_t o = (static_cast<size_t>(t0 + r) * H + h) * D + c4;
        va[it] = r < L ? ld4(src_a + o) : make_float4(0.f, 0.f, 0.f, 0.f);
        vb[it] = r < L ? ld4(src_b + o) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int e = tid + it * BT, r = e >> 5, c4 = (e & 31) * 4;
        *reinterpret_cast<float4*>(dst_a + r * LDW + c4) = va[it];
        *reinterpret_cast<float4*>(dst_b + r * LDW + c4) =
            make_float4(vb[it].x * scale_b, vb[it].y * scale_b, vb[it].z * scale_b, vb[it].w * scale_b);
    }
}

// State slabs through cp.async (16 bytes per copy), so that the next slab is in flight while the
// products read the current one.  Where a slab's rows must be scaled, each thread scales, after its
// own cp_wait, the very 16-byte chunks it copied (its own asynchronous writes are visible to it); the
// products that read the slab follow a __syncthreads.
// 32 rows i0 .. i0+31 of a state (stride 128) -> [32][LDW] tile
__device__ __forceinline__ void fetch_state_rows(float* dst, const float* S, int i0, int tid) {
#pragma unroll
    for (int it = 0; it < 32 * (D / 4) / BT; ++it) {
        const int e = tid + it * BT;
        cp16(dst + (e >> 5) * LDW + (e & 31) * 4, S + (i0 + (e >> 5)) * D + (e & 31) * 4);
    }
}
// row r of the slab times sc[i0 + r]
__device__ __forceinline__ void scale_state_rows(float* dst, int i0, const float* sc, int tid) {
#pragma unroll
    for (int it = 0; it < 32 * (D / 4) / BT; ++it) {
        const int e = tid + it * BT;
        float4* t = reinterpret_cast<float4*>(dst + (e >> 5) * LDW + (e & 31) * 4);
        const float f = sc[i0 + (e >> 5)];
        const float4 v = *t;
        *t = make_float4(v.x * f, v.y * f, v.z * f, v.w * f);
    }
}
// 32 columns j0 .. j0+31 of all 128 rows of a state -> [128][LDS] tile
__device__ __forceinline__ void fetch_state_cols(float* dst, const float* S, int j0, int tid) {
#pragma unroll
    for (int it = 0; it < D * 8 / BT; ++it) {
        const int e = tid + it * BT;
        cp16(dst + (e >> 3) * LDS + (e & 7) * 4, S + (e >> 3) * D + j0 + (e & 7) * 4);
    }
}

// Cumulative log-decay of the chunk in G: fetch_gates issues the cp.async copies of the log_alpha
// rows (rows >= L zero-filled; the caller commits, waits and synchronises the CTA), sum_gates sums
// down the rows (128 threads; rows >= L then hold gC) and writes e^{gm}, e^{gC - gm} (and e^{gC}) to
// vectors.  The caller synchronises the CTA after it.
__device__ __forceinline__ void fetch_gates(float* G, const float* la, int64_t t0, int L, int H, int h, int tid) {
    const float* row0 = la + (static_cast<size_t>(t0) * H + h) * D;
#pragma unroll
    for (int it = 0; it < C * (D / 4) / BT; ++it) {
        const int e = tid + it * BT, r = e >> 5, c4 = (e & 31) * 4;
        cp16z(G + r * LDW + c4, r < L ? row0 + static_cast<size_t>(r) * H * D + c4 : row0, r < L);
    }
}
__device__ __forceinline__ void sum_gates(float* G, int tid, float* egm, float* egcm, float* egc) {
    if (tid < D) {
        float s = 0.f, gm = 0.f;
#pragma unroll 8
        for (int r = 0; r < C; ++r) {
            s += G[r * LDW + tid];
            G[r * LDW + tid] = s;
            if (r == C / 2 - 1) gm = s;
        }
        egm[tid] = expf(gm);
        egcm[tid] = expf(s - gm);
        if (egc) egc[tid] = expf(s);
    }
}

// sequence of global chunk slot gc: the last n with chunk_off[n] <= gc
__device__ __forceinline__ int chunk_seq(const int32_t* chunk_off, int N, int gc) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= gc) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct ChunkPos {
    int n, c, L;
    int64_t t0;
};
__device__ __forceinline__ bool chunk_pos(const BackwardArgs& a, int gc, ChunkPos& p) {
    if (a.chunk_off[a.num_seqs + 1] == 0 || gc >= a.chunk_off[a.num_seqs]) return false;
    p.n = chunk_seq(a.chunk_off, a.num_seqs, gc);
    p.c = gc - a.chunk_off[p.n];
    p.t0 = static_cast<int64_t>(a.cu_seqlens[p.n]) + static_cast<int64_t>(p.c) * C;
    p.L = static_cast<int>(a.cu_seqlens[p.n + 1] - p.t0 < C ? a.cu_seqlens[p.n + 1] - p.t0 : C);
    return KDA_BOUNDS(p.n >= 0 && p.n < a.num_seqs && p.c >= 0 && gc < a.chunk_slots && p.t0 >= 0 && p.L >= 1 &&
                          p.t0 + p.L <= a.total_tokens,
                      a.device_status);
}
// state at the start of chunk (n, c): S0 (or zero) for the first chunk, else the snapshot after chunk c-1
__device__ __forceinline__ const float* chunk_start_state(const BackwardArgs& a, const ChunkPos& p, int gc, int h) {
    if (p.c == 0) return a.S0 ? a.S0 + (static_cast<size_t>(p.n) * a.H + h) * D * D : nullptr;
    return a.ckpt + (static_cast<size_t>(gc - 1) * a.H + h) * D * D;
}

// ================================================================ prep ==========
struct PrepL {
    static constexpr int KH = 0, QH = TILE, KB = 2 * TILE, DO = 3 * TILE;
    static constexpr int NF = 4 * TILE;          // [64][64] (m4 layout); NF..TF+4096 hold g first
    static constexpr int TF = NF + 4096;
    static constexpr int GS = NF;                // g scratch [64][LDW] spans NF, TF, XS and part of MM
    static constexpr int XS = TF + 4096;         // padding under the g scratch
    static constexpr int MM = XS + 768;
    static constexpr int TB = MM + PTILE;
    static constexpr int VB = TB + PTILE;        // beta[64], egm[128], egcm[128], egc[128]
    static constexpr int FLOATS = VB + 448;
};
static_assert(PrepL::GS + TILE <= PrepL::MM, "g scratch must end before Mm");
static_assert(PTILE >= pf::kInvScratchFloats, "the inverse's scratch fits the Tb tile");

template <typename IoT>
__global__ void __launch_bounds__(BT, 1) kda_bwd_prep_kernel(const BackwardArgs a) {
    extern __shared__ __align__(16) float sm[];
    using L = PrepL;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = 16 * (warp & 3), c64 = 32 * (warp >> 2), c128 = 64 * (warp >> 2);
    const int gc = blockIdx.x, h = blockIdx.y, H = a.H;
    ChunkPos p;
    if (!chunk_pos(a, gc, p)) return;
    const IoT* q = static_cast<const IoT*>(a.q);
    const IoT* k = static_cast<const IoT*>(a.k);
    float* rec = a.rec + (static_cast<size_t>(gc) * H + h) * kRecFloats;
    float *KH = sm + L::KH, *QH = sm + L::QH, *KB = sm + L::KB, *DO = sm + L::DO, *G = sm + L::GS;
    float *NF = sm + L::NF, *TF = sm + L::TF, *MM = sm + L::MM, *TB = sm + L::TB;
    float *bet = sm + L::VB, *egm = bet + 64, *egcm = egm + 128, *egc = egcm + 128;

    fetch_gates(G, a.log_alpha, p.t0, p.L, H, h, tid);
    cp_commit();
    load_tile2(KB, k, QH, q, p.t0, p.L, H, h, tid);
    load_tile(DO, static_cast<const IoT*>(a.dO), p.t0, p.L, H, h, tid);
    if (tid < C) bet[tid] = tid < p.L ? a.beta[(p.t0 + tid) * H + h] : 0.f;
    cp_wait<0>();
    __syncthreads();
    sum_gates(G, tid, egm, egcm, egc);
    __syncthreads();
    for (int e = tid; e < C * D; e += BT) {  // gated operands
        const int r = e >> 7, i = e & 127;
        const float x = G[r * LDW + i] - G[(C / 2 - 1) * LDW + i];
        const float ep = expf(x), en = expf(-x), kv = KB[r * LDW + i];
        KH[r * LDW + i] = kv * ep;
        KB[r * LDW + i] = kv * en;
        QH[r * LDW + i] *= ep;
    }
    __syncthreads();
    {   // Grams: N = Diag(beta) strict lower (Kh Kb^T) for the inverse; Mm = lower (Qh Kb^T)
        float ak[4][4], aq[4][4];
        zero(ak);
        zero(aq);
        mma16<4, AR, BN>(ak, KH, LDW, KB, LDW, D, r0, c64, lane);
        mma16<4, AR, BN>(aq, QH, LDW, KB, LDW, D, r0, c64, lane);
        __syncthreads();  // g scratch (over NF..MM) is dead
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = frow(r0, lane, e), s = fcol(c64, lane, j, e);
                pf::m1(NF, r, s) = s < r ? bet[r] * ak[j][e] : 0.f;
                MM[r * LDN + s] = s <= r ? aq[j][e] : 0.f;
            }
    }
    for (int e = tid; e < C * D; e += BT) {  // Kh Diag(e^{gm}) for the scan
        const int r = e >> 7, i = e & 127;
        rec[kRecKhm + e] = KH[r * LDW + i] * egm[i];
    }
    if (tid < D) rec[kRecGam + tid] = egc[tid];
    for (int half = 0; half < 2; ++half) {  // P = Diag(e^{gm}) Qh^T dO (128 x 128)
        float acc[8][4];
        zero(acc);
        mma16<8, AC, BK>(acc, QH + 64 * half, LDW, DO, LDW, C, r0, c128, lane);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {  // elements e, e + 1 are adjacent columns of one row
                const int i = 64 * half + frow(r0, lane, e), col = fcol(c128, lane, j, e);
                *reinterpret_cast<float2*>(rec + kRecP + i * D + col) =
                    make_float2(egm[i] * acc[j][e], egm[i] * acc[j][e + 1]);
            }
    }
    __syncthreads();
    // T = (I + N)^-1 (scratch in TB, written only after it), ends synchronised
    pf::lower_inverse_tc(pf::rows64(NF), pf::rows64(TF), TB, tid);
    for (int e = tid; e < C * C; e += BT) {
        const int r = e >> 6, s = e & 63;
        const float tb = s <= r ? pf::m1(TF, r, s) * bet[s] : 0.f;
        TB[r * LDN + s] = tb;
        rec[kRecTb + e] = tb;
    }
    __syncthreads();
    {   // Wbc = Tb^T Kb Diag(e^{gC-gm});  MdO = Mm^T dO (into QH)
        float acc[8][4], md[8][4];
        zero(acc);
        zero(md);
        mma16<8, AC, BK>(acc, TB, LDN, KB, LDW, C, r0, c128, lane);
        mma16<8, AC, BK>(md, MM, LDN, DO, LDW, C, r0, c128, lane);
        __syncthreads();  // QH is read no more
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int r = frow(r0, lane, e), i = fcol(c128, lane, j, e);
                *reinterpret_cast<float2*>(rec + kRecWbc + r * D + i) =
                    make_float2(acc[j][e] * egcm[i], acc[j][e + 1] * egcm[i + 1]);
                *reinterpret_cast<float2*>(QH + r * LDW + i) = make_float2(md[j][e], md[j][e + 1]);
            }
    }
    __syncthreads();
    {   // dY0 = -Tb^T MdO
        float acc[8][4];
        zero(acc);
        mma16<8, AC, BK>(acc, TB, LDN, QH, LDW, C, r0, c128, lane);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; e += 2)
                *reinterpret_cast<float2*>(rec + kRecDY0 + frow(r0, lane, e) * D + fcol(c128, lane, j, e)) =
                    make_float2(-acc[j][e], -acc[j][e + 1]);
    }
}

// ================================================================ scan ==========
// Per chunk (from the prep record): dY = dY0 - Wbc X;  X <- Diag(e^{gC}) X + P + Khm^T dY.
// The next chunk's record slices are prefetched (cp.async) while this one is computed.
struct ScanL {
    static constexpr int WB = 0;                 // [64][LDW]   Wbc
    static constexpr int KM = TILE;              // [64][LDW]   Khm
    static constexpr int PS = 2 * TILE;          // [128][LDX]  P, this CTA's columns
    static constexpr int Y0 = PS + 128 * LDX;    // [64][LDX]   dY0, this CTA's columns
    static constexpr int GM = Y0 + 64 * LDX;     // [128]       e^{gC}
    static constexpr int STAGE = GM + 128;
    static constexpr int XS = 2 * STAGE;         // [128][LDX]  X
    static constexpr int DY = XS + 128 * LDX;    // [64][LDS]   dY
    static constexpr int FLOATS = DY + 64 * LDS;
};
static_assert(ScanL::FLOATS * 4 <= 232448, "adjoint scan shared memory over the per-CTA limit");

__device__ __forceinline__ void scan_fetch(float* st, const float* rec, int c0, int tid) {
    for (int e = tid; e < C * (D / 4); e += BT) {
        const int r = e >> 5, c4 = (e & 31) * 4;
        cp16(st + ScanL::WB + r * LDW + c4, rec + kRecWbc + r * D + c4);
        cp16(st + ScanL::KM + r * LDW + c4, rec + kRecKhm + r * D + c4);
    }
    for (int e = tid; e < D * (NCS / 4); e += BT) {
        const int r = e >> 3, c4 = (e & 7) * 4;
        cp16(st + ScanL::PS + r * LDX + c4, rec + kRecP + r * D + c0 + c4);
        if (r < C) cp16(st + ScanL::Y0 + r * LDX + c4, rec + kRecDY0 + r * D + c0 + c4);
    }
    if (tid < D / 4) cp16(st + ScanL::GM + 4 * tid, rec + kRecGam + 4 * tid);
}

template <typename IoT>
__global__ void __launch_bounds__(BT, 1) kda_bwd_scan_kernel(const BackwardArgs a) {
    extern __shared__ __align__(16) float sm[];
    using L = ScanL;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, N = a.num_seqs;
    if (a.chunk_off[N + 1] == 0) return;
    const int unit = blockIdx.x;  // (rank of the sequence, longest first) x H x slices
    const int pos = unit / (H * kSlices);
    const int n = a.order ? a.order[pos] : pos, h = (unit / kSlices) % H, c0 = (unit % kSlices) * NCS;
    if (!KDA_BOUNDS(n >= 0 && n < N && h < H, a.device_status)) return;
    float *XS = sm + L::XS, *DY = sm + L::DY;
    const size_t sidx = (static_cast<size_t>(n) * H + h) * D * D;
    // X rows 16 warp + g (+8), columns 8 j + 2 t (+1) of this CTA's slice
    float X[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            X[j][e] = a.dS_final ? a.dS_final[sidx + frow(16 * warp, lane, e) * D + c0 + fcol(0, lane, j, e)] : 0.f;
    const int base = a.chunk_off[n], nch = a.chunk_off[n + 1] - base;
    const int64_t tb = a.cu_seqlens[n], te = a.cu_seqlens[n + 1];
    if (!KDA_BOUNDS(base >= 0 && nch >= 0 && base + nch <= a.chunk_slots && tb >= 0 && te >= tb &&
                        te <= a.total_tokens && static_cast<int64_t>(nch) * C >= te - tb &&
                        static_cast<int64_t>(nch) * C < te - tb + C,
                    a.device_status))
        return;
    auto rec_of = [&](int c) { return a.rec + (static_cast<size_t>(base + c) * H + h) * kRecFloats; };
    if (nch > 0) scan_fetch(sm, rec_of(nch - 1), c0, tid);
    cp_commit();
    for (int c = nch - 1, s = 0; c >= 0; --c, s ^= 1) {
        const int gc = base + c;
        const int64_t t0 = tb + static_cast<int64_t>(c) * C;
        const int Lr = static_cast<int>(te - t0 < C ? te - t0 : C);
        float* st = sm + s * L::STAGE;
        __syncthreads();  // the other stage and XS / DY are read no more
        if (c > 0) scan_fetch(sm + (s ^ 1) * L::STAGE, rec_of(c - 1), c0, tid);
        cp_commit();
        float* xo = a.xbuf + (static_cast<size_t>(gc) * H + h) * D * D;
        // the state after this chunk at this thread's X elements, in flight until the X update
        float sn[4][4];
        {
            const float* snp = a.ckpt + (static_cast<size_t>(gc) * H + h) * D * D + c0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const float2 v = *reinterpret_cast<const float2*>(snp + frow(16 * warp, lane, e) * D +
                                                                      fcol(0, lane, j, e));
                    sn[j][e] = v.x;
                    sn[j][e + 1] = v.y;
                }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {  // elements e, e + 1 are adjacent columns of one row
                const int r = frow(16 * warp, lane, e), col = fcol(0, lane, j, e);
                *reinterpret_cast<float2*>(XS + r * LDX + col) = make_float2(X[j][e], X[j][e + 1]);
            }
        cp_wait<1>();  // this chunk's stage has landed
        __syncthreads();
        // the adjoint of this chunk's end state, as whole 128-byte row segments of the slice
        for (int e = tid; e < D * (NCS / 4); e += BT) {
            const int r = e / (NCS / 4), c4 = 4 * (e % (NCS / 4));
            *reinterpret_cast<float4*>(xo + r * D + c0 + c4) = *reinterpret_cast<const float4*>(XS + r * LDX + c4);
        }
        {   // dY = dY0 - Wbc X  (64 x 32: warp rows 16 (warp & 3), columns 16 (warp >> 2))
            const int r0 = 16 * (warp & 3), cc = 16 * (warp >> 2);
            float acc[2][4];
            zero(acc);
            mma16<2, AR, BK8>(acc, st + L::WB, LDW, XS, LDX, D, r0, cc, lane);
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = frow(r0, lane, e), col = fcol(cc, lane, j, e);
                    const float2 y0 = *reinterpret_cast<const float2*>(st + L::Y0 + r * LDX + col);
                    DY[r * LDS + col] = y0.x - acc[j][e];
                    DY[r * LDS + col + 1] = y0.y - acc[j][e + 1];
                }
        }
        __syncthreads();
        for (int e = tid; e < Lr * (NCS / 4); e += BT) {  // dv = -dY, whole row segments of the slice
            const int r = e / (NCS / 4), c4 = 4 * (e % (NCS / 4));
            const float4 dy = *reinterpret_cast<const float4*>(DY + r * LDS + c4);
            *reinterpret_cast<float4*>(a.dv + (static_cast<size_t>(t0 + r) * H + h) * D + c0 + c4) =
                make_float4(-dy.x, -dy.y, -dy.z, -dy.w);
        }
        {   // this slice's part of rowsum(S_next * X), the last row's boundary term of dlog_alpha, into
            // row i >> 5, column c0 + (i & 31) of the record's P block (consumed: the stage holds it)
            float p_lo = 0.f, p_hi = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                p_lo = fmaf(sn[j][0], X[j][0], fmaf(sn[j][1], X[j][1], p_lo));
                p_hi = fmaf(sn[j][2], X[j][2], fmaf(sn[j][3], X[j][3], p_hi));
            }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                p_lo += __shfl_xor_sync(0xffffffffu, p_lo, off);
                p_hi += __shfl_xor_sync(0xffffffffu, p_hi, off);
            }
            if ((lane & 3) == 0) {
                float* bp = rec_of(c) + kRecP + c0;
                const int i_lo = frow(16 * warp, lane, 0), i_hi = i_lo + 8;
                bp[(i_lo >> 5) * D + (i_lo & 31)] = p_lo;
                bp[(i_hi >> 5) * D + (i_hi & 31)] = p_hi;
            }
        }
        {   // X <- Diag(e^{gC}) X + P + Khm^T dY
            float acc[4][4];
            zero(acc);
            mma16<4, AC, BK>(acc, st + L::KM, LDW, DY, LDS, C, 16 * warp, 0, lane);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int r = frow(16 * warp, lane, e), col = fcol(0, lane, j, e);
                    const float2 ps = *reinterpret_cast<const float2*>(st + L::PS + r * LDX + col);
                    const float gm = st[L::GM + r];
                    X[j][e] = fmaf(gm, X[j][e], ps.x + acc[j][e]);
                    X[j][e + 1] = fmaf(gm, X[j][e + 1], ps.y + acc[j][e + 1]);
                }
        }
    }
    cp_wait<0>();
    if (a.dS0) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                a.dS0[sidx + frow(16 * warp, lane, e) * D + c0 + fcol(0, lane, j, e)] = X[j][e];
    }
}

// ========================================================== value + key =========
// One CTA per (chunk, head) runs the value products (U, R, du, dbeta) and then the key products (dq, dk,
// dlog alpha): U, dO and dY stay in shared memory between them instead of a round trip through global
// memory, and the chunk's q, k, log alpha and states are fetched by one CTA, not two.
struct ValueKeyL {
    static constexpr int T0 = 0, T1 = TILE, T2 = 2 * TILE, T3 = 3 * TILE;
    static constexpr int P0 = 4 * TILE, P1 = P0 + PTILE;
    // two slab buffers: [32][LDW] row slabs of a state (value phase), [128][LDS] column slabs (key
    // phase); ST2 holds Tb [64][LDN] between the start-state and adjoint slabs
    static constexpr int ST = P1 + PTILE;
    static constexpr int ST2 = ST + 128 * LDS;
    static constexpr int VB = ST2 + 128 * LDS;   // egm[128], egcm[128], dbeta halves [2][64] / boundary terms
    static constexpr int FLOATS = VB + 384;
};
static_assert(32 * LDW <= 128 * LDS && C * LDN <= 128 * LDS, "the value phase's slabs fit the ST slot");
static_assert(ValueKeyL::ST % 4 == 0 && ValueKeyL::ST2 % 4 == 0, "16-byte aligned slab buffers");
static_assert(ValueKeyL::FLOATS * 4 <= 232448, "value+key shared memory over the per-CTA limit");

// The key products of one (chunk, head), with dO in T0, U in T1 and dY in T2 already resident; T3
// takes the gates, ST and ST2 the state and adjoint column slabs ([128][LDS]), two in flight at a
// time.  Ends with dq, dk, dlog alpha.
template <typename IoT>
__device__ __forceinline__ void key_phase(const BackwardArgs& a, const ChunkPos& p, int gc, int h, float* T0, float* T1,
                                          float* T2, float* T3, float* P0, float* P1, float* ST, float* ST2,
                                          float* egm, float* egcm, float* bnd, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    const int r0 = 16 * (warp & 3), c64 = 32 * (warp >> 2), c128 = 64 * (warp >> 2);
    const int H = a.H;
    const IoT* q = static_cast<const IoT*>(a.q);
    const IoT* k = static_cast<const IoT*>(a.k);
    const float* X = a.xbuf + (static_cast<size_t>(gc) * H + h) * D * D;
    const float* S = chunk_start_state(a, p, gc, h);
    // column slabs: those of the start state (dO Sm^T, dY Sm^T; none when it is zero), then the
    // adjoint's (U Xc^T); the first two are fetched while the gates and the triangular products run
    const int nslab = S ? 8 : 4;
    auto slab_src = [&](int i) { return (S && i < 4) ? S : X; };
    fetch_state_cols(ST, slab_src(0), 0, tid);
    cp_commit();
    fetch_state_cols(ST2, slab_src(1), 32, tid);
    cp_commit();
    load_tile(T3, a.log_alpha, p.t0, p.L, H, h, tid);
    __syncthreads();
    sum_gates(T3, tid, egm, egcm, nullptr);
    if (tid < D) {  // boundary term of the last row, rowsum(S_next * X): the adjoint scan's four slice parts
        const float* bp = a.rec + (static_cast<size_t>(gc) * H + h) * kRecFloats + kRecP + (tid >> 5) * D + (tid & 31);
        bnd[tid] = (bp[0] + bp[NCS]) + (bp[2 * NCS] + bp[3 * NCS]);
    }
    __syncthreads();
    {   // P0 = lower (dO U^T) incl. diagonal; P1 = strict upper (U dY^T)
        float a0[4][4], a1[4][4];
        zero(a0);
        zero(a1);
        mma16<4, AR, BN>(a0, T0, LDW, T1, LDW, D, r0, c64, lane);
        mma16<4, AR, BN>(a1, T1, LDW, T2, LDW, D, r0, c64, lane);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = frow(r0, lane, e), s = fcol(c64, lane, j, e);
                P0[r * LDN + s] = s <= r ? a0[j][e] : 0.f;
                P1[r * LDN + s] = s > r ? a1[j][e] : 0.f;
            }
    }
    float aq[8][4], aka[8][4], akb[8][4];
    zero(aq);
    zero(aka);
    zero(akb);
    // dO S^T, dY S^T; then U X^T (states in 32-column slabs).  The row scalings of Sm = Diag(e^{gm}) S
    // and Xc = Diag(e^{gC-gm}) X scale the products' output columns, so they are applied to the
    // accumulators afterwards instead of to every slab.
    for (int i = 0; i < nslab; ++i) {
        float* buf = (i & 1) ? ST2 : ST;
        const bool of_s = S && i < 4;
        const int j0 = 32 * (i & 3);
        cp_wait<1>();  // slab i has landed (slab i + 1 may be in flight)
        __syncthreads();
        if (of_s) {
            mma16<8, AR, BN>(aq, T0 + j0, LDW, buf, LDS, 32, r0, c128, lane);
            mma16<8, AR, BN>(akb, T2 + j0, LDW, buf, LDS, 32, r0, c128, lane);
        } else {
            mma16<8, AR, BN>(aka, T1 + j0, LDW, buf, LDS, 32, r0, c128, lane);
        }
        __syncthreads();  // buf is read no more
        if (i + 2 < nslab) fetch_state_cols(buf, slab_src(i + 2), 32 * ((i + 2) & 3), tid);
        cp_commit();
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = fcol(c128, lane, j, e);
            aq[j][e] *= egm[i];
            akb[j][e] *= egm[i];
            aka[j][e] *= egcm[i];
        }
    // dO, U, dY are read no more
    load_tile2(T2, k, T1, q, p.t0, p.L, H, h, tid);
    __syncthreads();
    for (int e = tid; e < C * D; e += BT) {  // T0 = Kh, T1 = Qh, T2 = Kb
        const int r = e >> 7, i = e & 127;
        const float x = T3[r * LDW + i] - T3[(C / 2 - 1) * LDW + i];
        const float ep = expf(x), kv = T2[r * LDW + i];
        T0[r * LDW + i] = kv * ep;
        T2[r * LDW + i] = kv * expf(-x);
        T1[r * LDW + i] *= ep;
    }
    __syncthreads();
    mma16<8, AR, BK>(aq, P0, LDN, T2, LDW, C, r0, c128, lane);   // tril(dO U^T) Kb
    mma16<8, AC, BK>(aka, P0, LDN, T1, LDW, C, r0, c128, lane);  // triu(U dO^T) Qh
    mma16<8, AR, BK>(aka, P1, LDN, T0, LDW, C, r0, c128, lane);  // striu(U dY^T) Kh
    mma16<8, AC, BK>(akb, P1, LDN, T2, LDW, C, r0, c128, lane);  // stril(dY U^T) Kb
    __syncthreads();  // T0 takes dg
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {  // elements e, e + 1 are adjacent columns of one row
            const int r = frow(r0, lane, e), i = fcol(c128, lane, j, e);
            float dq[2], dk[2], dg[2] = {0.f, 0.f}, dd[2], qv[2], kv[2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const float gx = T3[r * LDW + i + x] - T3[(C / 2 - 1) * LDW + i + x];
                const float eq = expf(gx), eb = expf(-gx);
                const float dka = eb * aka[j][e + x], dkb = eq * akb[j][e + x];
                dq[x] = eq * aq[j][e + x];
                dk[x] = dka + dkb;
                dd[x] = dkb - dka;
                // q and k back from the gated tiles (Qh = q e^{g-gm}, Kb = k e^{gm-g}), to fp32 rounding
                qv[x] = T1[r * LDW + i + x] * eb;
                kv[x] = T2[r * LDW + i + x] * eq;
            }
            if (r < p.L) {
                const size_t o = (static_cast<size_t>(p.t0 + r) * H + h) * D + i;
                dg[0] = qv[0] * dq[0] + kv[0] * dd[0];
                dg[1] = qv[1] * dq[1] + kv[1] * dd[1];
                if (r == p.L - 1) {
                    dg[0] += bnd[i];
                    dg[1] += bnd[i + 1];
                }
                *reinterpret_cast<float2*>(a.dq + o) = make_float2(dq[0], dq[1]);
                *reinterpret_cast<float2*>(a.dk + o) = make_float2(dk[0], dk[1]);
            }
            *reinterpret_cast<float2*>(T0 + r * LDW + i) = make_float2(dg[0], dg[1]);
        }
    __syncthreads();
    if (tid < D) {  // dlog_alpha = reverse cumulative sum of dg
        float s = 0.f;
        for (int r = p.L - 1; r >= 0; --r) {
            s += T0[r * LDW + tid];
            a.dla[(static_cast<size_t>(p.t0 + r) * H + h) * D + tid] = s;
        }
    }
}


template <typename IoT>
__global__ void __launch_bounds__(BT, 1) kda_bwd_value_key_kernel(const BackwardArgs a) {
    extern __shared__ __align__(16) float sm[];
    using L = ValueKeyL;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = 16 * (warp & 3), c64 = 32 * (warp >> 2), c128 = 64 * (warp >> 2);
    const int gc = blockIdx.x, h = blockIdx.y, H = a.H;
    ChunkPos p;
    if (!chunk_pos(a, gc, p)) return;
    float *T0 = sm + L::T0, *T1 = sm + L::T1, *T2 = sm + L::T2, *T3 = sm + L::T3, *P0 = sm + L::P0,
          *P1 = sm + L::P1, *ST = sm + L::ST, *ST2 = sm + L::ST2, *egm = sm + L::VB, *egcm = egm + 128,
          *dbh = egcm + 128;
    const IoT* k = static_cast<const IoT*>(a.k);
    const float* S = chunk_start_state(a, p, gc, h);
    const float* X = a.xbuf + (static_cast<size_t>(gc) * H + h) * D * D;
    // the log_alpha rows, then the start state's first two 32-row slabs are in flight while k and q
    // load and the gates and Grams are formed
    fetch_gates(T3, a.log_alpha, p.t0, p.L, H, h, tid);
    cp_commit();
    if (S) {
        fetch_state_rows(ST, S, 0, tid);
        cp_commit();
        fetch_state_rows(ST2, S, 32, tid);
        cp_commit();
    }
    load_tile2(T1, k, T2, static_cast<const IoT*>(a.q), p.t0, p.L, H, h, tid);
    if (S) cp_wait<2>();
    else cp_wait<0>();
    __syncthreads();
    sum_gates(T3, tid, egm, egcm, nullptr);
    __syncthreads();
    for (int e = tid; e < C * D; e += BT) {  // T0 = Kh, T1 = Kb, T2 = Qh
        const int r = e >> 7, i = e & 127;
        const float x = T3[r * LDW + i] - T3[(C / 2 - 1) * LDW + i];
        const float ep = expf(x), kv = T1[r * LDW + i];
        T0[r * LDW + i] = kv * ep;
        T1[r * LDW + i] = kv * expf(-x);
        T2[r * LDW + i] *= ep;
    }
    __syncthreads();
    {   // P0 = Lm = strict lower (Kh Kb^T), P1 = Mm = lower (Qh Kb^T)
        float al[4][4], am[4][4];
        zero(al);
        zero(am);
        mma16<4, AR, BN>(al, T0, LDW, T1, LDW, D, r0, c64, lane);
        mma16<4, AR, BN>(am, T2, LDW, T1, LDW, D, r0, c64, lane);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = frow(r0, lane, e), s = fcol(c64, lane, j, e);
                P0[r * LDN + s] = s < r ? al[j][e] : 0.f;
                P1[r * LDN + s] = s <= r ? am[j][e] : 0.f;
            }
    }
    // Kh Sm, the start state streamed in 32-row slabs, two in flight
    float acc[8][4];
    zero(acc);
    if (S) {
        for (int i = 0; i < D / 32; ++i) {
            float* buf = (i & 1) ? ST2 : ST;
            cp_wait<1>();  // slab i has landed (slab i + 1 may be in flight)
            scale_state_rows(buf, 32 * i, egm, tid);
            __syncthreads();
            mma16<8, AR, BK>(acc, T0 + 32 * i, LDW, buf, LDW, 32, r0, c128, lane);
            __syncthreads();  // buf is read no more
            if (i + 2 < D / 32) fetch_state_rows(buf, S, 32 * (i + 2), tid);
            cp_commit();
        }
    }
    __syncthreads();  // T2 (Qh), ST and ST2 are read no more
    {   // Tb -> ST2 and the adjoint's first slab -> ST, in flight while v loads
        const float* tbg = a.rec + (static_cast<size_t>(gc) * H + h) * kRecFloats + kRecTb;
#pragma unroll
        for (int it = 0; it < C * (C / 4) / BT; ++it) {
            const int e = tid + it * BT, r = e >> 4, c4 = (e & 15) * 4;
            cp16(ST2 + r * LDN + c4, tbg + r * C + c4);
        }
        cp_commit();
        fetch_state_rows(ST, X, 0, tid);
        cp_commit();
    }
    load_tile(T2, static_cast<const IoT*>(a.v), p.t0, p.L, H, h, tid);
    cp_wait<1>();  // Tb has landed
    __syncthreads();
    float rr[8][4];  // Y1 = V - Kh Sm (own elements), later R
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = frow(r0, lane, e), i = fcol(c128, lane, j, e);
            rr[j][e] = T2[r * LDW + i] - acc[j][e];
        }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) T2[frow(r0, lane, e) * LDW + fcol(c128, lane, j, e)] = rr[j][e];
    __syncthreads();
    zero(acc);
    mma16<8, AR, BK>(acc, ST2, LDN, T2, LDW, C, r0, c128, lane);  // U = Tb Y1
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {  // elements e, e + 1 are adjacent columns of one row
            const int r = frow(r0, lane, e), i = fcol(c128, lane, j, e);
            const float2 u = make_float2(acc[j][e], acc[j][e + 1]);
            *reinterpret_cast<float2*>(T3 + r * LDW + i) = u;  // U stays in T3 for the key phase
        }
    __syncthreads();
    zero(acc);
    mma16<8, AR, BK>(acc, P0, LDN, T3, LDW, C, r0, c128, lane);  // Lm U
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) rr[j][e] -= acc[j][e];  // R
    __syncthreads();  // T0 (Kh), T2 and ST2 (Tb) are read no more
    fetch_state_rows(ST2, X, 32, tid);
    cp_commit();
    load_tile(T2, static_cast<const IoT*>(a.dO), p.t0, p.L, H, h, tid);
    load_tile(T0, a.dv, p.t0, p.L, H, h, tid, -1.f);  // dY = -dv
    __syncthreads();
    zero(acc);
    mma16<8, AC, BK>(acc, P1, LDN, T2, LDW, C, r0, c128, lane);  // Mm^T dO
    mma16<8, AC, BK>(acc, P0, LDN, T0, LDW, C, r0, c128, lane);  // + Lm^T dY
    for (int i = 0; i < D / 32; ++i) {  // + Kb Xc, X streamed in 32-row slabs, two in flight
        float* buf = (i & 1) ? ST2 : ST;
        cp_wait<1>();
        scale_state_rows(buf, 32 * i, egcm, tid);
        __syncthreads();
        mma16<8, AR, BK>(acc, T1 + 32 * i, LDW, buf, LDW, 32, r0, c128, lane);
        __syncthreads();  // buf is read no more
        if (i + 2 < D / 32) fetch_state_rows(buf, X, 32 * (i + 2), tid);
        cp_commit();
    }
    // dbeta_t = <du_t, r_t>: rows g, g + 8 of the warp; columns over the 4 threads of a group
    // and the two warps (warp, warp + 4) that share the rows
    float s_lo = 0.f, s_hi = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        s_lo = fmaf(acc[j][0], rr[j][0], fmaf(acc[j][1], rr[j][1], s_lo));
        s_hi = fmaf(acc[j][2], rr[j][2], fmaf(acc[j][3], rr[j][3], s_hi));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        s_lo += __shfl_xor_sync(0xffffffffu, s_lo, off);
        s_hi += __shfl_xor_sync(0xffffffffu, s_hi, off);
    }
    if ((lane & 3) == 0) {
        dbh[(warp >> 2) * 64 + frow(r0, lane, 0)] = s_lo;
        dbh[(warp >> 2) * 64 + frow(r0, lane, 2)] = s_hi;
    }
    __syncthreads();
    if (tid < p.L) a.dbeta[(p.t0 + tid) * H + h] = dbh[tid] + dbh[64 + tid];
    __syncthreads();  // dbh, Kb (T1), Mm and Lm are read no more

    // ---- key phase: dq, dk, dlog alpha.  dO (T2), U (T3) and dY (T0) are resident; the tiles are
    // renamed to the key products' roles: K0 = dO, K1 = U, K2 = dY, K3 = the gates (into Kb's tile)
    key_phase<IoT>(a, p, gc, h, T2, T3, T0, T1, P0, P1, ST, ST2, egm, egcm, egcm + 128, tid);
}

// ============================================================ fused prologue ==
// kda_prefill_backward_ex: the prologue of "kimi delta attn from first principles" (aryagxr),
// "KDA Architecture" (q, k L2-normalised) and "KDA has three gates" (beta = sigmoid of its
// projection) is applied to copies before the backward, and differentiated after it:
//   x_hat = x s, s = 1 / sqrt(sum_c x_c^2 + eps):  dx = s (dx_hat - x_hat <x_hat, dx_hat>)
//   beta = sigmoid(b):                             db = dbeta beta (1 - beta)
// One warp per (token, head) row; x_hat is recomputed in fp32 from the original x.
template <typename IoT>
__global__ void kda_bwd_prologue_kernel(const IoT* __restrict__ q, const IoT* __restrict__ k,
                                        const float* __restrict__ beta, IoT* __restrict__ qh, IoT* __restrict__ kh,
                                        float* __restrict__ bh, float* __restrict__ inv, int64_t rows, uint32_t flags,
                                        float eps) {
    const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    if (flags & KDA_FUSE_L2NORM_QK) {
        const size_t o = static_cast<size_t>(row) * D + 4 * lane;
        const float4 qv = ld4(q + o), kv = ld4(k + o);
        float aq = qv.x * qv.x + qv.y * qv.y + qv.z * qv.z + qv.w * qv.w;
        float ak = kv.x * kv.x + kv.y * kv.y + kv.z * kv.z + kv.w * kv.w;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            aq += __shfl_xor_sync(0xffffffffu, aq, off);
            ak += __shfl_xor_sync(0xffffffffu, ak, off);
        }
        const float sq = 1.f / sqrtf(aq + eps), sk = 1.f / sqrtf(ak + eps);
        st4(qh + o, make_float4(qv.x * sq, qv.y * sq, qv.z * sq, qv.w * sq));
        st4(kh + o, make_float4(kv.x * sk, kv.y * sk, kv.z * sk, kv.w * sk));
        if (lane == 0) *reinterpret_cast<float2*>(inv + 2 * row) = make_float2(sq, sk);
    }
    if ((flags & KDA_FUSE_BETA_SIGMOID) && lane == 0) bh[row] = 1.f / (1.f + expf(-beta[row]));
}

template <typename IoT>
__global__ void kda_bwd_epilogue_kernel(const IoT* __restrict__ q, const IoT* __restrict__ k,
                                        const float* __restrict__ bh, const float* __restrict__ inv,
                                        float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dbeta,
                                        int64_t rows, uint32_t flags) {
    const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    if (flags & KDA_FUSE_L2NORM_QK) {
        const size_t o = static_cast<size_t>(row) * D + 4 * lane;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const float s = inv[2 * row + w];
            const float4 x = ld4((w == 0 ? q : k) + o);
            float* g = (w == 0 ? dq : dk) + o;
            const float4 d = *reinterpret_cast<const float4*>(g);
            const float4 xh = make_float4(x.x * s, x.y * s, x.z * s, x.w * s);
            float dot = xh.x * d.x + xh.y * d.y + xh.z * d.z + xh.w * d.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            *reinterpret_cast<float4*>(g) = make_float4(s * (d.x - xh.x * dot), s * (d.y - xh.y * dot),
                                                        s * (d.z - xh.z * dot), s * (d.w - xh.w * dot));
        }
    }
    if ((flags & KDA_FUSE_BETA_SIGMOID) && lane == 0) {
        const float b = bh[row];
        dbeta[row] *= b * (1.f - b);
    }
}

// ============================================================== output gate ==
// kda_prefill_backward_gated: the output gate of "kimi delta attn from first principles" (aryagxr),
// "KDA has three gates", y = o r w g with r = (sum_j o_j^2 / 128 + eps)^(-1/2), differentiated for
// L = <y, dY>:
//   do_m = r w_m g_m dY_m - (r^3 o_m / 128) sum_j dY_j o_j w_j g_j,   dg_j = dY_j o_j r w_j,
//   dw_j = sum over (token, head) rows of dY_j o_j r g_j.
// One warp per (token, head) row, 4 channels per lane, rows grid-strided over a fixed grid so that
// dw's per-block partial sums (and their fixed-order sum in kda_bwd_outgate_sum_kernel) are
// bitwise repeatable.  do is written in the input dtype (the chunkwise backward reads dO in it); it may
// overwrite o in place, since each warp holds its whole row in registers before it stores.
constexpr int kGateBlocks = 592;  // 4 x 148 blocks of 8 warps

template <typename IoT>
__global__ void __launch_bounds__(256) kda_bwd_outgate_kernel(const IoT* o, const IoT* __restrict__ g,
                                                              const IoT* __restrict__ dy,
                                                              const float* __restrict__ w, float eps,
                                                              IoT* dout, float* __restrict__ dg,
                                                              float* __restrict__ dw_part, int64_t rows) {
    __shared__ float4 part[8][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 wv = w ? make_float4(w[4 * lane], w[4 * lane + 1], w[4 * lane + 2], w[4 * lane + 3])
                        : make_float4(1.f, 1.f, 1.f, 1.f);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp; row < rows;
         row += static_cast<int64_t>(gridDim.x) * 8) {
        const size_t off = static_cast<size_t>(row) * D + 4 * lane;
        const float4 ov = ld4(o + off), gv = ld4(g + off), yv = ld4(dy + off);
        const float4 a = make_float4(wv.x * gv.x * yv.x, wv.y * gv.y * yv.y, wv.z * gv.z * yv.z, wv.w * gv.w * yv.w);
        float ss = ov.x * ov.x + ov.y * ov.y + ov.z * ov.z + ov.w * ov.w;
        float dot = a.x * ov.x + a.y * ov.y + a.z * ov.z + a.w * ov.w;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, sh);
            dot += __shfl_xor_sync(0xffffffffu, dot, sh);
        }
        const float r = rsqrtf(ss * (1.f / D) + eps);
        const float c = r * r * r * (1.f / D) * dot;
        st4(dout + off, make_float4(r * a.x - c * ov.x, r * a.y - c * ov.y, r * a.z - c * ov.z, r * a.w - c * ov.w));
        *reinterpret_cast<float4*>(dg + off) =
            make_float4(yv.x * ov.x * r * wv.x, yv.y * ov.y * r * wv.y, yv.z * ov.z * r * wv.z, yv.w * ov.w * r * wv.w);
        acc.x = fmaf(yv.x * ov.x, r * gv.x, acc.x);
        acc.y = fmaf(yv.y * ov.y, r * gv.y, acc.y);
        acc.z = fmaf(yv.z * ov.z, r * gv.z, acc.z);
        acc.w = fmaf(yv.w * ov.w, r * gv.w, acc.w);
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float4 t = part[0][lane];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            const float4 u = part[i][lane];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        *reinterpret_cast<float4*>(dw_part + static_cast<size_t>(blockIdx.x) * D + 4 * lane) = t;
    }
}

// dw = the sum of the per-block partials, in block order (one thread per channel).
__global__ void kda_bwd_outgate_sum_kernel(const float* __restrict__ dw_part, int nparts, float* __restrict__ dw) {
    const int c = threadIdx.x;
    float t = 0.f;
    for (int b = 0; b < nparts; ++b) t += dw_part[static_cast<size_t>(b) * D + c];
    dw[c] = t;
}

// Snapshot entries for every chunk end of every sequence: entry chunk_off[n] + c - 1 is the state
// after chunk c - 1 of sequence n (c = 1 .. nch_n; the last is the final state).  Entries past the
// batch's chunk count are sentinels (sequence N) that no scan CTA takes.
__global__ void kda_ckpt_entries_kernel(const int32_t* __restrict__ cu_seqlens,
                                        const int32_t* __restrict__ chunk_off, int32_t N, int32_t max_entries,
                                        int32_t* __restrict__ snap_seq, int32_t* __restrict__ snap_pos,
                                        int32_t* device_status) {
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
    if (!KDA_BOUNDS(base >= 0 && nch >= 0 && base + nch <= max_entries, device_status)) return;
    for (int c = 1; c <= nch; ++c) {
        snap_seq[base + c - 1] = n;
        snap_pos[base + c - 1] = min(c * C, len);
    }
}

template <typename K>
cudaError_t launch_smem(K kern, dim3 grid, size_t smem, const BackwardArgs& a, cudaStream_t stream) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    kern<<<grid, BT, smem, stream>>>(a);
    return cudaGetLastError();
}

template <typename IoT>
cudaError_t launch_all(const BackwardArgs& a, int64_t chunk_slots, cudaStream_t stream) {
    const dim3 per_chunk(static_cast<unsigned>(chunk_slots), static_cast<unsigned>(a.H));
    cudaError_t err;
    if ((err = launch_smem(kda_bwd_prep_kernel<IoT>, per_chunk, PrepL::FLOATS * 4, a, stream)) != cudaSuccess)
        return err;
    const unsigned scan_ctas = static_cast<unsigned>(a.num_seqs) * a.H * kSlices;
    if (scan_ctas > 0 &&
        (err = launch_smem(kda_bwd_scan_kernel<IoT>, dim3(scan_ctas), ScanL::FLOATS * 4, a, stream)) != cudaSuccess)
        return err;
    return launch_smem(kda_bwd_value_key_kernel<IoT>, per_chunk, ValueKeyL::FLOATS * 4, a, stream);
}

}  // namespace

size_t backward_record_bytes() { return static_cast<size_t>(kRecFloats) * 4; }

cudaError_t launch_ckpt_entries(const int32_t* cu_seqlens, const int32_t* chunk_off, int32_t N, int32_t max_entries,
                                int32_t* snap_seq, int32_t* snap_pos, int32_t* device_status, cudaStream_t stream) {
    const int threads = 128, blocks = (N + 1 + threads - 1) / threads;
    kda_ckpt_entries_kernel<<<blocks, threads, 0, stream>>>(cu_seqlens, chunk_off, N, max_entries, snap_seq,
                                                            snap_pos, device_status);
    return cudaGetLastError();
}

cudaError_t launch_bwd_prologue(bool f32_io, const void* q, const void* k, const float* beta, void* qh, void* kh,
                                float* bh, float* inv, int64_t rows, uint32_t flags, float eps, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    if (f32_io)
        kda_bwd_prologue_kernel<float><<<blocks, 256, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), beta, static_cast<float*>(qh),
            static_cast<float*>(kh), bh, inv, rows, flags, eps);
    else
        kda_bwd_prologue_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), beta,
            static_cast<__nv_bfloat16*>(qh), static_cast<__nv_bfloat16*>(kh), bh, inv, rows, flags, eps);
    return cudaGetLastError();
}

cudaError_t launch_bwd_epilogue(bool f32_io, const void* q, const void* k, const float* bh, const float* inv,
                                float* dq, float* dk, float* dbeta, int64_t rows, uint32_t flags,
                                cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    if (f32_io)
        kda_bwd_epilogue_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float*>(q),
                                                                   static_cast<const float*>(k), bh, inv, dq, dk,
                                                                   dbeta, rows, flags);
    else
        kda_bwd_epilogue_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), bh, inv, dq, dk, dbeta,
            rows, flags);
    return cudaGetLastError();
}

size_t outgate_partial_bytes() { return static_cast<size_t>(kGateBlocks) * D * 4; }

cudaError_t launch_bwd_outgate(bool f32_io, const void* o, const void* g, const void* dy, const float* w, float eps,
                               void* dout, float* dg, float* dw, float* dw_part, int64_t rows, cudaStream_t stream) {
    if (rows > 0) {
        if (f32_io)
            kda_bwd_outgate_kernel<float><<<kGateBlocks, 256, 0, stream>>>(
                static_cast<const float*>(o), static_cast<const float*>(g), static_cast<const float*>(dy), w, eps,
                static_cast<float*>(dout), dg, dw_part, rows);
        else
            kda_bwd_outgate_kernel<__nv_bfloat16><<<kGateBlocks, 256, 0, stream>>>(
                static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(g),
                static_cast<const __nv_bfloat16*>(dy), w, eps, static_cast<__nv_bfloat16*>(dout), dg, dw_part, rows);
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    if (dw) {
        if (rows > 0) kda_bwd_outgate_sum_kernel<<<1, D, 0, stream>>>(dw_part, kGateBlocks, dw);
        else if (cudaMemsetAsync(dw, 0, D * sizeof(float), stream) != cudaSuccess) return cudaGetLastError();
    }
    return cudaGetLastError();
}

cudaError_t launch_backward(const BackwardArgs& a, bool f32_io, int64_t chunk_slots, cudaStream_t stream) {
    if (chunk_slots <= 0 || a.H <= 0) return cudaSuccess;
    return f32_io ? launch_all<float>(a, chunk_slots, stream) : launch_all<__nv_bfloat16>(a, chunk_slots, stream);
}

}  // namespace kda
