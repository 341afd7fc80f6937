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
// Kernels (all 256 threads, fp32 products on the CUDA cores from shared memory):
//   prep      per (chunk, head): the X-independent pieces -> a per-chunk record
//   scan      per (sequence, head, 32 state columns): the walk of X; writes dv = -dY
//             and X after every chunk
//   value     per (chunk, head): U (kept in the grad_q buffer until the key kernel), dbeta
//   key       per (chunk, head): dq, dk, dlog_alpha
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
constexpr int TILE = C * LDW;
constexpr int PTILE = C * LDN;
constexpr int NCS = 32;       // state columns per scan CTA
constexpr int kSlices = D / NCS;

// per-(chunk, head) record of the prep kernel (fp32)
constexpr int kRecWbc = 0;        // [64][128] Tb^T Kb Diag(e^{gC-gm})
constexpr int kRecDY0 = 8192;     // [64][128] -Tb^T Mm^T dO
constexpr int kRecQhm = 16384;    // [64][128] Qh Diag(e^{gm})
constexpr int kRecKhm = 24576;    // [64][128] Kh Diag(e^{gm})
constexpr int kRecTb = 32768;     // [64][64]  Tb
constexpr int kRecGam = 36864;    // [128]     e^{gC}
constexpr int kRecFloats = 36992;

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
__device__ __forceinline__ float ld1(const T* p);
template <>
__device__ __forceinline__ float ld1<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float comp(const float4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// ---- products on shared tiles ---------------------------------------------------------------
// Every product accumulates a 64-row output in the same thread layout: thread (rb = tid >> 4,
// cb = tid & 15) owns rows 4 rb + y (y < 4) and columns cb + 16 x (x < NX).
//   nn: C += A B     A[m][k] (k contiguous), B[k][n] (n contiguous)
//   tn: C += At^T B  At[k][m], B[k][n]
//   nt: C += A Bt^T  A[m][k], Bt[n][k]   (Bt's stride = 4 mod 32 floats)
template <int NX>
__device__ __forceinline__ void g_nn(float (&acc)[4][NX], const float* A, int lda, const float* B, int ldb, int K,
                                     int rb, int cb) {
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float4 a[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) a[y] = *reinterpret_cast<const float4*>(A + (4 * rb + y) * lda + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float b[NX];
#pragma unroll
            for (int x = 0; x < NX; ++x) b[x] = B[(k + kk) * ldb + cb + 16 * x];
#pragma unroll
            for (int y = 0; y < 4; ++y)
#pragma unroll
                for (int x = 0; x < NX; ++x) acc[y][x] = fmaf(comp(a[y], kk), b[x], acc[y][x]);
        }
    }
}
template <int NX>
__device__ __forceinline__ void g_tn(float (&acc)[4][NX], const float* At, int lda, const float* B, int ldb, int K,
                                     int rb, int cb) {
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        const float4 a = *reinterpret_cast<const float4*>(At + k * lda + 4 * rb);
        float b[NX];
#pragma unroll
        for (int x = 0; x < NX; ++x) b[x] = B[k * ldb + cb + 16 * x];
#pragma unroll
        for (int x = 0; x < NX; ++x) {
            acc[0][x] = fmaf(a.x, b[x], acc[0][x]);
            acc[1][x] = fmaf(a.y, b[x], acc[1][x]);
            acc[2][x] = fmaf(a.z, b[x], acc[2][x]);
            acc[3][x] = fmaf(a.w, b[x], acc[3][x]);
        }
    }
}
template <int NX>
__device__ __forceinline__ void g_nt(float (&acc)[4][NX], const float* A, int lda, const float* Bt, int ldb, int K,
                                     int rb, int cb) {
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float4 a[4], b[NX];
#pragma unroll
        for (int y = 0; y < 4; ++y) a[y] = *reinterpret_cast<const float4*>(A + (4 * rb + y) * lda + k);
#pragma unroll
        for (int x = 0; x < NX; ++x) b[x] = *reinterpret_cast<const float4*>(Bt + (cb + 16 * x) * ldb + k);
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int x = 0; x < NX; ++x) {
                float s = acc[y][x];
                s = fmaf(a[y].x, b[x].x, s);
                s = fmaf(a[y].y, b[x].y, s);
                s = fmaf(a[y].z, b[x].z, s);
                s = fmaf(a[y].w, b[x].w, s);
                acc[y][x] = s;
            }
    }
}
template <int NX>
__device__ __forceinline__ void zero(float (&acc)[4][NX]) {
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < NX; ++x) acc[y][x] = 0.f;
}

// ---- loads ------------------------------------------------------------------------------------
// rows [t0, t0 + L) of a [T, H, 128] tensor, head h -> fp32 tile (stride LDW), rows >= L zero
template <typename T>
__device__ __forceinline__ void load_tile(float* dst, const T* src, int64_t t0, int L, int H, int h, int tid,
                                          float scale = 1.f) {
    for (int e = tid; e < C * (D / 4); e += BT) {
        const int r = e >> 5, c4 = (e & 31) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < L) {
            v = ld4(src + (static_cast<size_t>(t0 + r) * H + h) * D + c4);
            v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
        }
        *reinterpret_cast<float4*>(dst + r * LDW + c4) = v;
    }
}
// [64][128] fp32 record section -> tile (stride LDW)
__device__ __forceinline__ void load_rec(float* dst, const float* src, int tid) {
    for (int e = tid; e < C * (D / 4); e += BT) {
        const int r = e >> 5, c4 = (e & 31) * 4;
        *reinterpret_cast<float4*>(dst + r * LDW + c4) = *reinterpret_cast<const float4*>(src + r * D + c4);
    }
}

// cumulative log-decay of the chunk (rows >= L hold gC), by 128 threads; e^{gm}, e^{gC - gm} to vectors
__device__ __forceinline__ void chunk_gates(float* G, const float* la, int64_t t0, int L, int H, int h, int tid,
                                            float* egm, float* egcm, float* egc) {
    if (tid < D) {
        float s = 0.f, gm = 0.f;
        for (int r = 0; r < C; ++r) {
            if (r < L) s += la[(static_cast<size_t>(t0 + r) * H + h) * D + tid];
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
    return true;
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
    static constexpr int XS = TF + 4096;
    static constexpr int MM = XS + 768;
    static constexpr int TB = MM + PTILE;
    static constexpr int VB = TB + PTILE;        // beta[64], egm[128], egcm[128], egc[128]
    static constexpr int FLOATS = VB + 448;
};
static_assert(PrepL::GS + TILE <= PrepL::MM, "g scratch must end before Mm");

template <typename IoT>
__global__ void __launch_bounds__(BT, 1) kda_bwd_prep_kernel(const BackwardArgs a) {
    extern __shared__ __align__(16) float sm[];
    using L = PrepL;
    const int tid = threadIdx.x, rb = tid >> 4, cb = tid & 15;
    const int gc = blockIdx.x, h = blockIdx.y, H = a.H;
    ChunkPos p;
    if (!chunk_pos(a, gc, p)) return;
    const IoT* q = static_cast<const IoT*>(a.q);
    const IoT* k = static_cast<const IoT*>(a.k);
    float* rec = a.rec + (static_cast<size_t>(gc) * H + h) * kRecFloats;
    float *KH = sm + L::KH, *QH = sm + L::QH, *KB = sm + L::KB, *DO = sm + L::DO, *G = sm + L::GS;
    float *NF = sm + L::NF, *TF = sm + L::TF, *XS = sm + L::XS, *MM = sm + L::MM, *TB = sm + L::TB;
    float *bet = sm + L::VB, *egm = bet + 64, *egcm = egm + 128, *egc = egcm + 128;

    load_tile(KB, k, p.t0, p.L, H, h, tid);
    load_tile(QH, q, p.t0, p.L, H, h, tid);
    load_tile(DO, static_cast<const IoT*>(a.dO), p.t0, p.L, H, h, tid);
    chunk_gates(G, a.log_alpha, p.t0, p.L, H, h, tid, egm, egcm, egc);
    if (tid < C) bet[tid] = tid < p.L ? a.beta[(p.t0 + tid) * H + h] : 0.f;
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
        g_nt<4>(ak, KH, LDW, KB, LDW, D, rb, cb);
        g_nt<4>(aq, QH, LDW, KB, LDW, D, rb, cb);
        __syncthreads();  // g scratch (over NF..MM) is dead
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int r = 4 * rb + y, s = cb + 16 * x;
                pf::m1(NF, r, s) = s < r ? bet[r] * ak[y][x] : 0.f;
                MM[r * LDN + s] = s <= r ? aq[y][x] : 0.f;
            }
    }
    for (int e = tid; e < C * D; e += BT) {  // Qh, Kh scaled by e^{gm} for the scan
        const int r = e >> 7, i = e & 127;
        rec[kRecQhm + e] = QH[r * LDW + i] * egm[i];
        rec[kRecKhm + e] = KH[r * LDW + i] * egm[i];
    }
    if (tid < D) rec[kRecGam + tid] = egc[tid];
    __syncthreads();
    pf::lower_inverse(NF, TF, XS, tid);  // T = (I + N)^-1, ends synchronised
    for (int e = tid; e < C * C; e += BT) {
        const int r = e >> 6, s = e & 63;
        const float tb = s <= r ? pf::m1(TF, r, s) * bet[s] : 0.f;
        TB[r * LDN + s] = tb;
        rec[kRecTb + e] = tb;
    }
    __syncthreads();
    {   // Wbc = Tb^T Kb Diag(e^{gC-gm});  MdO = Mm^T dO (into QH)
        float acc[4][8], md[4][8];
        zero(acc);
        zero(md);
        g_tn<8>(acc, TB, LDN, KB, LDW, C, rb, cb);
        g_tn<8>(md, MM, LDN, DO, LDW, C, rb, cb);
        __syncthreads();  // QH is read no more
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const int r = 4 * rb + y, i = cb + 16 * x;
                rec[kRecWbc + r * D + i] = acc[y][x] * egcm[i];
                QH[r * LDW + i] = md[y][x];
            }
    }
    __syncthreads();
    {   // dY0 = -Tb^T MdO
        float acc[4][8];
        zero(acc);
        g_tn<8>(acc, TB, LDN, QH, LDW, C, rb, cb);
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int x = 0; x < 8; ++x) rec[kRecDY0 + (4 * rb + y) * D + cb + 16 * x] = -acc[y][x];
    }
}

// ================================================================ scan ==========
struct ScanL {
    static constexpr int WB = 0;                 // [64][LDW]   Wbc
    static constexpr int QK = TILE;              // [128][LDW]  [Qhm; Khm]
    static constexpr int BB = QK + 2 * TILE;     // [128][LDS]  [dO; dY] (this CTA's columns)
    static constexpr int Y0 = BB + 128 * LDS;    // [64][LDS]   dY0
    static constexpr int XS = Y0 + 64 * LDS;     // [128][LDS]  X
    static constexpr int GM = XS + 128 * LDS;    // [128]       e^{gC}
    static constexpr int FLOATS = GM + 128;
};

template <typename IoT>
__global__ void __launch_bounds__(BT, 1) kda_bwd_scan_kernel(const BackwardArgs a) {
    extern __shared__ __align__(16) float sm[];
    using L = ScanL;
    const int tid = threadIdx.x, rb = tid >> 4, cb = tid & 15;
    const int H = a.H, N = a.num_seqs;
    if (a.chunk_off[N + 1] == 0) return;
    const int unit = blockIdx.x;  // (rank of the sequence, longest first) x H x slices
    const int n = a.order[unit / (H * kSlices)], h = (unit / kSlices) % H, c0 = (unit % kSlices) * NCS;
    float *WB = sm + L::WB, *QK = sm + L::QK, *BB = sm + L::BB, *Y0 = sm + L::Y0, *XS = sm + L::XS,
          *GM = sm + L::GM;
    const size_t sidx = (static_cast<size_t>(n) * H + h) * D * D;
    float X[2][4][2];  // rows 64 z + 4 rb + y, columns c0 + cb + 16 x
#pragma unroll
    for (int z = 0; z < 2; ++z)
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int x = 0; x < 2; ++x)
                X[z][y][x] = a.dS_final ? a.dS_final[sidx + (64 * z + 4 * rb + y) * D + c0 + cb + 16 * x] : 0.f;
    const int base = a.chunk_off[n], nch = a.chunk_off[n + 1] - base;
    const int64_t tb = a.cu_seqlens[n], te = a.cu_seqlens[n + 1];
    for (int c = nch - 1; c >= 0; --c) {
        const int gc = base + c;
        const int64_t t0 = tb + static_cast<int64_t>(c) * C;
        const int Lr = static_cast<int>(te - t0 < C ? te - t0 : C);
        const float* rec = a.rec + (static_cast<size_t>(gc) * H + h) * kRecFloats;
        __syncthreads();  // the previous chunk's shared data is read no more
        float* xo = a.xbuf + (static_cast<size_t>(gc) * H + h) * D * D;
#pragma unroll
        for (int z = 0; z < 2; ++z)
#pragma unroll
            for (int y = 0; y < 4; ++y)
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int r = 64 * z + 4 * rb + y, col = cb + 16 * x;
                    XS[r * LDS + col] = X[z][y][x];
                    xo[r * D + c0 + col] = X[z][y][x];
                }
        load_rec(WB, rec + kRecWbc, tid);
        load_rec(QK, rec + kRecQhm, tid);
        load_rec(QK + TILE, rec + kRecKhm, tid);
        for (int e = tid; e < C * (NCS / 4); e += BT) {
            const int r = e >> 3, c4 = (e & 7) * 4;
            *reinterpret_cast<float4*>(Y0 + r * LDS + c4) =
                *reinterpret_cast<const float4*>(rec + kRecDY0 + r * D + c0 + c4);
            float4 d = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < Lr) d = ld4(static_cast<const IoT*>(a.dO) + (static_cast<size_t>(t0 + r) * H + h) * D + c0 + c4);
            *reinterpret_cast<float4*>(BB + r * LDS + c4) = d;
        }
        if (tid < D) GM[tid] = rec[kRecGam + tid];
        __syncthreads();
        {   // dY = dY0 - Wbc X
            float acc[4][2];
            zero(acc);
            g_nn<2>(acc, WB, LDW, XS, LDS, D, rb, cb);
#pragma unroll
            for (int y = 0; y < 4; ++y)
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int r = 4 * rb + y, col = cb + 16 * x;
                    const float dy = Y0[r * LDS + col] - acc[y][x];
                    BB[(C + r) * LDS + col] = dy;
                    if (r < Lr) a.dv[(static_cast<size_t>(t0 + r) * H + h) * D + c0 + col] = -dy;
                }
        }
        __syncthreads();
        {   // X <- Diag(e^{gC}) X + [Qhm; Khm]^T [dO; dY]
            float lo[4][2], hi[4][2];
            zero(lo);
            zero(hi);
            g_tn<2>(lo, QK, LDW, BB, LDS, 2 * C, rb, cb);
            g_tn<2>(hi, QK + 64, LDW, BB, LDS, 2 * C, rb, cb);
#pragma unroll
            for (int y = 0; y < 4; ++y)
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    X[0][y][x] = fmaf(GM[4 * rb + y], X[0][y][x], lo[y][x]);
                    X[1][y][x] = fmaf(GM[64 + 4 * rb + y], X[1][y][x], hi[y][x]);
                }
        }
    }
    if (a.dS0) {
#pragma unroll
        for (int z = 0; z < 2; ++z)
#pragma unroll
            for (int y = 0; y < 4; ++y)
#pragma unroll
                for (int x = 0; x < 2; ++x) a.dS0[sidx + (64 * z + 4 * rb + y) * D + c0 + cb + 16 * x] = X[z][y][x];
    }
}

// ================================================================ value =========
struct ValueL {
    static constexpr int T0 = 0, T1 = TILE, T2 = 2 * TILE, T3 = 3 * TILE;
    static constexpr int P0 = 4 * TILE, P1 = P0 + PTILE;
    static constexpr int ST = P1 + PTILE;        // [32][LDW] state slab, or Tb [64][LDN]
    static constexpr int VB = ST + PTILE;        // egm[128], egcm[128]
    static constexpr int FLOATS = VB + 256;
};
static_assert(32 * LDW <= PTILE, "state slab fits the Tb slot");

template <typename IoT>
__global__ void __launch_bounds__(BT, 1) kda_bwd_value_kernel(const BackwardArgs a) {
    extern __shared__ __align__(16) float sm[];
    using L = ValueL;
    const int tid = threadIdx.x, rb = tid >> 4, cb = tid & 15;
    const int gc = blockIdx.x, h = blockIdx.y, H = a.H;
    ChunkPos p;
    if (!chunk_pos(a, gc, p)) return;
    float *T0 = sm + L::T0, *T1 = sm + L::T1, *T2 = sm + L::T2, *T3 = sm + L::T3, *P0 = sm + L::P0,
          *P1 = sm + L::P1, *ST = sm + L::ST, *egm = sm + L::VB, *egcm = egm + 128;
    const IoT* k = static_cast<const IoT*>(a.k);

    load_tile(T1, k, p.t0, p.L, H, h, tid);
    load_tile(T2, static_cast<const IoT*>(a.q), p.t0, p.L, H, h, tid);
    chunk_gates(T3, a.log_alpha, p.t0, p.L, H, h, tid, egm, egcm, nullptr);
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
        g_nt<4>(al, T0, LDW, T1, LDW, D, rb, cb);
        g_nt<4>(am, T2, LDW, T1, LDW, D, rb, cb);
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int r = 4 * rb + y, s = cb + 16 * x;
                P0[r * LDN + s] = s < r ? al[y][x] : 0.f;
                P1[r * LDN + s] = s <= r ? am[y][x] : 0.f;
            }
    }
    // Kh Sm, the start state streamed in 32-row slabs
    float acc[4][8];
    zero(acc);
    const float* S = chunk_start_state(a, p, gc, h);
    if (S) {
        for (int i0 = 0; i0 < D; i0 += 32) {
            __syncthreads();
            for (int e = tid; e < 32 * (D / 4); e += BT) {
                const int r = e >> 5, c4 = (e & 31) * 4;
                float4 v = *reinterpret_cast<const float4*>(S + (i0 + r) * D + c4);
                const float s = egm[i0 + r];
                v.x *= s; v.y *= s; v.z *= s; v.w *= s;
                *reinterpret_cast<float4*>(ST + r * LDW + c4) = v;
            }
            __syncthreads();
            g_nn<8>(acc, T0 + i0, LDW, ST, LDW, 32, rb, cb);
        }
    }
    __syncthreads();  // T2 (Qh) and ST are read no more
    load_tile(T2, static_cast<const IoT*>(a.v), p.t0, p.L, H, h, tid);
    {
        const float* tbg = a.rec + (static_cast<size_t>(gc) * H + h) * kRecFloats + kRecTb;
        for (int e = tid; e < C * (C / 4); e += BT) {
            const int r = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(ST + r * LDN + c4) = *reinterpret_cast<const float4*>(tbg + r * C + c4);
        }
    }
    __syncthreads();
    float rr[4][8];  // Y1 = V - Kh Sm (own elements), later R
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int r = 4 * rb + y, i = cb + 16 * x;
            rr[y][x] = T2[r * LDW + i] - acc[y][x];
        }
    __syncthreads();
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 8; ++x) T2[(4 * rb + y) * LDW + cb + 16 * x] = rr[y][x];
    __syncthreads();
    zero(acc);
    g_nn<8>(acc, ST, LDN, T2, LDW, C, rb, cb);  // U = Tb Y1
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int r = 4 * rb + y, i = cb + 16 * x;
            T3[r * LDW + i] = acc[y][x];
            if (r < p.L) a.u_scratch[(static_cast<size_t>(p.t0 + r) * H + h) * D + i] = acc[y][x];
        }
    __syncthreads();
    zero(acc);
    g_nn<8>(acc, P0, LDN, T3, LDW, C, rb, cb);  // Lm U
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 8; ++x) rr[y][x] -= acc[y][x];  // R
    __syncthreads();  // T2, T3 and ST are read no more
    load_tile(T2, static_cast<const IoT*>(a.dO), p.t0, p.L, H, h, tid);
    load_tile(T3, a.dv, p.t0, p.L, H, h, tid, -1.f);  // dY = -dv
    __syncthreads();
    zero(acc);
    g_tn<8>(acc, P1, LDN, T2, LDW, C, rb, cb);  // Mm^T dO
    g_tn<8>(acc, P0, LDN, T3, LDW, C, rb, cb);  // + Lm^T dY
    {   // + Kb Xc, X streamed in 32-row slabs
        const float* X = a.xbuf + (static_cast<size_t>(gc) * H + h) * D * D;
        for (int i0 = 0; i0 < D; i0 += 32) {
            __syncthreads();
            for (int e = tid; e < 32 * (D / 4); e += BT) {
                const int r = e >> 5, c4 = (e & 31) * 4;
                float4 v = *reinterpret_cast<const float4*>(X + (i0 + r) * D + c4);
                const float s = egcm[i0 + r];
                v.x *= s; v.y *= s; v.z *= s; v.w *= s;
                *reinterpret_cast<float4*>(ST + r * LDW + c4) = v;
            }
            __syncthreads();
            g_nn<8>(acc, T1 + i0, LDW, ST, LDW, 32, rb, cb);
        }
    }
    // dbeta_t = <du_t, r_t>: the 16 threads of a row group share the rows
#pragma unroll
    for (int y = 0; y < 4; ++y) {
        float s = 0.f;
#pragma unroll
        for (int x = 0; x < 8; ++x) s = fmaf(acc[y][x], rr[y][x], s);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const int r = 4 * rb + y;
        if (cb == 0 && r < p.L) a.dbeta[(p.t0 + r) * H + h] = s;
    }
}

// ================================================================ key ===========
struct KeyL {
    static constexpr int T0 = 0, T1 = TILE, T2 = 2 * TILE, T3 = 3 * TILE;
    static constexpr int P0 = 4 * TILE, P1 = P0 + PTILE;
    static constexpr int ST = P1 + PTILE;        // [128][LDS] state column slab
    static constexpr int VB = ST + 128 * LDS;    // egm[128], egcm[128], bnd[128]
    static constexpr int FLOATS = VB + 384;
};

template <typename IoT>
__global__ void __launch_bounds__(BT, 1) kda_bwd_key_kernel(const BackwardArgs a) {
    extern __shared__ __align__(16) float sm[];
    using L = KeyL;
    const int tid = threadIdx.x, rb = tid >> 4, cb = tid & 15;
    const int gc = blockIdx.x, h = blockIdx.y, H = a.H;
    ChunkPos p;
    if (!chunk_pos(a, gc, p)) return;
    float *T0 = sm + L::T0, *T1 = sm + L::T1, *T2 = sm + L::T2, *T3 = sm + L::T3, *P0 = sm + L::P0,
          *P1 = sm + L::P1, *ST = sm + L::ST, *egm = sm + L::VB, *egcm = egm + 128, *bnd = egcm + 128;
    const IoT* q = static_cast<const IoT*>(a.q);
    const IoT* k = static_cast<const IoT*>(a.k);
    const float* X = a.xbuf + (static_cast<size_t>(gc) * H + h) * D * D;

    load_tile(T0, static_cast<const IoT*>(a.dO), p.t0, p.L, H, h, tid);
    load_tile(T1, a.u_scratch, p.t0, p.L, H, h, tid);
    load_tile(T2, a.dv, p.t0, p.L, H, h, tid, -1.f);  // dY
    chunk_gates(T3, a.log_alpha, p.t0, p.L, H, h, tid, egm, egcm, nullptr);
    {   // boundary term of the last row: rowsum(S_next * X), S_next = the snapshot after this chunk
        const float* Sn = a.ckpt + (static_cast<size_t>(gc) * H + h) * D * D;
        const int i = tid >> 1, j0 = (tid & 1) * 64;
        float s = 0.f;
        for (int j = 0; j < 64; j += 4) {
            const float4 sv = *reinterpret_cast<const float4*>(Sn + i * D + j0 + j);
            const float4 xv = *reinterpret_cast<const float4*>(X + i * D + j0 + j);
            s = fmaf(sv.x, xv.x, fmaf(sv.y, xv.y, fmaf(sv.z, xv.z, fmaf(sv.w, xv.w, s))));
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        if ((tid & 1) == 0) bnd[i] = s;
    }
    __syncthreads();
    {   // P0 = lower (dO U^T) incl. diagonal; P1 = strict upper (U dY^T)
        float a0[4][4], a1[4][4];
        zero(a0);
        zero(a1);
        g_nt<4>(a0, T0, LDW, T1, LDW, D, rb, cb);
        g_nt<4>(a1, T1, LDW, T2, LDW, D, rb, cb);
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int r = 4 * rb + y, s = cb + 16 * x;
                P0[r * LDN + s] = s <= r ? a0[y][x] : 0.f;
                P1[r * LDN + s] = s > r ? a1[y][x] : 0.f;
            }
    }
    float aq[4][8], aka[4][8], akb[4][8];
    zero(aq);
    zero(aka);
    zero(akb);
    const float* S = chunk_start_state(a, p, gc, h);
    for (int pass = 0; pass < 2; ++pass) {  // dO Sm^T, dY Sm^T; then U Xc^T (states in 32-column slabs)
        const float* M = pass == 0 ? S : X;
        if (!M) continue;
        const float* sc = pass == 0 ? egm : egcm;
        for (int j0 = 0; j0 < D; j0 += 32) {
            __syncthreads();
            for (int e = tid; e < D * 8; e += BT) {
                const int i = e >> 3, c4 = (e & 7) * 4;
                float4 v = *reinterpret_cast<const float4*>(M + i * D + j0 + c4);
                const float s = sc[i];
                v.x *= s; v.y *= s; v.z *= s; v.w *= s;
                *reinterpret_cast<float4*>(ST + i * LDS + c4) = v;
            }
            __syncthreads();
            if (pass == 0) {
                g_nt<8>(aq, T0 + j0, LDW, ST, LDS, 32, rb, cb);
                g_nt<8>(akb, T2 + j0, LDW, ST, LDS, 32, rb, cb);
            } else {
                g_nt<8>(aka, T1 + j0, LDW, ST, LDS, 32, rb, cb);
            }
        }
    }
    __syncthreads();  // dO, U, dY are read no more
    load_tile(T2, k, p.t0, p.L, H, h, tid);
    load_tile(T1, q, p.t0, p.L, H, h, tid);
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
    g_nn<8>(aq, P0, LDN, T2, LDW, C, rb, cb);   // tril(dO U^T) Kb
    g_tn<8>(aka, P0, LDN, T1, LDW, C, rb, cb);  // triu(U dO^T) Qh
    g_nn<8>(aka, P1, LDN, T0, LDW, C, rb, cb);  // striu(U dY^T) Kh
    g_tn<8>(akb, P1, LDN, T2, LDW, C, rb, cb);  // stril(dY U^T) Kb
    __syncthreads();  // T0 takes dg
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int r = 4 * rb + y, i = cb + 16 * x;
            const float gx = T3[r * LDW + i] - T3[(C / 2 - 1) * LDW + i];
            const float eq = expf(gx), eb = expf(-gx);
            const float dq = eq * aq[y][x], dka = eb * aka[y][x], dkb = eq * akb[y][x];
            float dg = 0.f;
            if (r < p.L) {
                const size_t o = (static_cast<size_t>(p.t0 + r) * H + h) * D + i;
                dg = ld1(q + o) * dq + ld1(k + o) * (dkb - dka);
                if (r == p.L - 1) dg += bnd[i];
                a.dq[o] = dq;
                a.dk[o] = dka + dkb;
            }
            T0[r * LDW + i] = dg;
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
    if ((err = launch_smem(kda_bwd_value_kernel<IoT>, per_chunk, ValueL::FLOATS * 4, a, stream)) != cudaSuccess)
        return err;
    return launch_smem(kda_bwd_key_kernel<IoT>, per_chunk, KeyL::FLOATS * 4, a, stream);
}

}  // namespace

size_t backward_record_bytes() { return static_cast<size_t>(kRecFloats) * 4; }

cudaError_t launch_ckpt_entries(const int32_t* cu_seqlens, const int32_t* chunk_off, int32_t N, int32_t max_entries,
                                int32_t* snap_seq, int32_t* snap_pos, cudaStream_t stream) {
    const int threads = 128, blocks = (N + 1 + threads - 1) / threads;
    kda_ckpt_entries_kernel<<<blocks, threads, 0, stream>>>(cu_seqlens, chunk_off, N, max_entries, snap_seq,
                                                            snap_pos);
    return cudaGetLastError();
}

cudaError_t launch_backward(const BackwardArgs& a, bool f32_io, int64_t chunk_slots, cudaStream_t stream) {
    if (chunk_slots <= 0 || a.H <= 0) return cudaSuccess;
    return f32_io ? launch_all<float>(a, chunk_slots, stream) : launch_all<__nv_bfloat16>(a, chunk_slots, stream);
}

}  // namespace kda
