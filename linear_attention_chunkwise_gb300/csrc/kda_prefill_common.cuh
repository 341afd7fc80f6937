// kda_prefill_common.cuh -- device code shared by the prefill kernels: the
// per-chunk gate phase, the triangular inverse, TMEM/packing helpers.
//
// Chunk algebra (derived from the KDA equation of "Understanding Kimi Delta
// Attention" (pyshine), section "The KDA Recurrence", and o_t = S_t^T q_t of
// "kimi delta attn from first principles" (aryagxr), section "KDA"), per chunk
// of C = 64 rows with start state S (dk x dv, rows = key channels):
//   g   = inclusive cumsum of log_alpha over the chunk rows (per channel)
//   gm  = g at row 31 (reference row), gC = g at row 63
//   Kh  = k*exp(g-gm),  Qh = q*exp(g-gm),  Kb = k*exp(gm-g)            (bf16)
//   A   = Kh Kb^T (strictly lower part),  M = lower(Qh Kb^T) (incl. diagonal)
//   T   = (I + Diag(beta) A)^-1,  Tb = T Diag(beta)
//   W   = Tb Kh,  U0 = Tb V,  Sm = Diag(exp(gm)) S
//   U   = U0 - W Sm,  O = Qh Sm + M U
//   S  <- Diag(exp(gC)) S + Diag(exp(gC-gm)) Kb^T U
// Rows past the sequence end are masked to k = q = v = 0, beta = 0,
// log_alpha = 0, which makes them exact no-ops.
#pragma once

#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {
namespace pf {

constexpr int C = kChunk;    // 64
constexpr int D = kHeadDim;  // 128
constexpr int NT = 256;      // threads per CTA
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t tmem_lane(int quarter) { return static_cast<uint32_t>(32 * quarter) << 16; }

// 2^x with the hardware approximation (relative error ~2^-22); exp(y) is
// evaluated as 2^(y log2 e).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// fp32 [64][64] scratch with the float4 column index xor-swizzled by the row
// (conflict-free row-per-thread and column-per-thread accesses).
__device__ __forceinline__ float4& m4(float* M, int r, int c4) {
    return *reinterpret_cast<float4*>(M + r * 64 + (((c4 ^ r) & 15) << 2));
}
__device__ __forceinline__ float& m1(float* M, int r, int c) {
    return M[r * 64 + ((((c >> 2) ^ r) & 15) << 2) + (c & 3)];
}
// The same [64][64] scratch with rows 0..31 at `lo` and rows 32..63 at `hi` (two separate 8 KB
// regions, e.g. the halves of a tile that has already been stored).
struct Rows64 {
    float* lo;
    float* hi;
};
__device__ __forceinline__ Rows64 rows64(float* M) { return Rows64{M, M + 32 * 64}; }
__device__ __forceinline__ float* row_of(const Rows64& M, int r) {
    return (r < 32 ? M.lo : M.hi) + (r & 31) * 64;
}
__device__ __forceinline__ float4& m4(const Rows64& M, int r, int c4) {
    return *reinterpret_cast<float4*>(row_of(M, r) + (((c4 ^ r) & 15) << 2));
}
__device__ __forceinline__ float& m1(const Rows64& M, int r, int c) {
    return row_of(M, r)[((((c >> 2) ^ r) & 15) << 2) + (c & 3)];
}

__device__ __forceinline__ uint4 pack8(const float* v) {
    uint4 pk;
    pk.x = pack_bf16(v[0], v[1]);
    pk.y = pack_bf16(v[2], v[3]);
    pk.z = pack_bf16(v[4], v[5]);
    pk.w = pack_bf16(v[6], v[7]);
    return pk;
}

template <typename OutT>
__device__ __forceinline__ void store_out8(OutT* dst, const float* v);
template <>
__device__ __forceinline__ void store_out8<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
    *reinterpret_cast<uint4*>(dst) = pack8(v);
}
template <>
__device__ __forceinline__ void store_out8<float>(float* dst, const float* v) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ float4 fma4(float s, const float4& a, const float4& acc) {
    return make_float4(fmaf(s, a.x, acc.x), fmaf(s, a.y, acc.y), fmaf(s, a.z, acc.z), fmaf(s, a.w, acc.w));
}

// log_alpha of the rows this thread handles in the gate phase (rows 16 (tid / 64) .. +15, channels
// 2 (tid % 64), +1; zero past row Lc), from shared or global memory with `stride` floats per row.
__device__ __forceinline__ void gate_load(const float* la, int stride, int Lc, int tid, float (&g0)[16],
                                          float (&g1)[16]) {
    const int cp = tid & 63, rq = tid >> 6;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = 16 * rq + i;
        float2 l2 = make_float2(0.f, 0.f);
        if (r < Lc) l2 = *reinterpret_cast<const float2*>(la + static_cast<size_t>(r) * stride + 2 * cp);
        g0[i] = l2.x;
        g1[i] = l2.y;
    }
}

// Gate phase of one chunk (all NT threads; one __syncthreads inside).
//   g0/g1: this thread's log_alpha values from gate_load (overwritten)
//   opa  : operand tile [2 blk][128 rows][128 B]; rows 0..63 hold k and rows
//          64..127 hold q on entry (128B-swizzled bf16), Kh and Qh on exit
//   opkb : [2 blk][64 rows][128 B], receives Kb
//   Lc   : valid rows of the chunk; red: f32 [4][128] scratch
//   beta_s[64] receives beta (masked) from beta_cur of threads 0..63
//   egm/egc/egcm[128] receive exp(gm), exp(gC), exp(gC - gm) per channel
__device__ __forceinline__ void gate_chunk(float (&g0)[16], float (&g1)[16], uint8_t* opa, uint8_t* opkb, int Lc,
                                           float* red, float* beta_s, float beta_cur, float* egm, float* egc,
                                           float* egcm, int tid, const float* inv_norm = nullptr) {
    const int cp = tid & 63;  // channel pair (2cp, 2cp+1)
    const int rq = tid >> 6;  // rows 16rq .. 16rq+15
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        acc0 += g0[i];
        acc1 += g1[i];
        g0[i] = acc0;
        g1[i] = acc1;
    }
    reinterpret_cast<float2*>(red + rq * D)[cp] = make_float2(acc0, acc1);
    if (tid < C) beta_s[tid] = (tid < Lc) ? beta_cur : 0.f;
    __syncthreads();
    float2 part[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) part[qq] = reinterpret_cast<const float2*>(red + qq * D)[cp];
    float off0 = 0.f, off1 = 0.f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
        if (qq < rq) { off0 += part[qq].x; off1 += part[qq].y; }
    const float gm0 = part[0].x + part[1].x, gm1 = part[0].y + part[1].y;
    const float gC0 = gm0 + part[2].x + part[3].x, gC1 = gm1 + part[2].y + part[3].y;
    if (rq == 0) {
        egm[2 * cp] = expf(gm0); egm[2 * cp + 1] = expf(gm1);
        egc[2 * cp] = expf(gC0); egc[2 * cp + 1] = expf(gC1);
        egcm[2 * cp] = expf(gC0 - gm0); egcm[2 * cp + 1] = expf(gC1 - gm1);
    }
    const float c0 = (off0 - gm0) * kLog2e, c1 = (off1 - gm1) * kLog2e;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = 16 * rq + i;
        const float x0 = fmaf(g0[i], kLog2e, c0), x1 = fmaf(g1[i], kLog2e, c1);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
        const float f0 = ex2_approx(-x0), f1 = ex2_approx(-x1);
        const uint32_t koff = sw128_off(r, 2 * cp, 16384);
        const uint32_t qoff = sw128_off(64 + r, 2 * cp, 16384);
        float2 kk = make_float2(0.f, 0.f), qv = kk;
        if (r < Lc) {
            kk = unpack_bf16(*reinterpret_cast<const uint32_t*>(opa + koff));
            qv = unpack_bf16(*reinterpret_cast<const uint32_t*>(opa + qoff));
            if (inv_norm) {  // fused L2 normalisation of k and q rows
                const float ik = inv_norm[r], iq = inv_norm[64 + r];
                kk.x *= ik; kk.y *= ik; qv.x *= iq; qv.y *= iq;
            }
        }
        *reinterpret_cast<uint32_t*>(opa + koff) = pack_bf16(kk.x * e0, kk.y * e1);
        *reinterpret_cast<uint32_t*>(opa + qoff) = pack_bf16(qv.x * e0, qv.y * e1);
        *reinterpret_cast<uint32_t*>(opkb + sw128_off(r, 2 * cp, 8192)) = pack_bf16(kk.x * f0, kk.y * f1);
    }
}

// The gate phase with 4 channels x 8 rows per thread: thread tid handles channels 4 (tid % 32) .. +3
// of rows 8 (tid / 32) .. +7, so a warp covers one 8-row group across all 128 channels (whole
// 512-byte rows of log_alpha per load, conflict-free 8-byte tile accesses, and a quarter of the
// address arithmetic per channel of gate_chunk).  Same results as gate_chunk.
__device__ __forceinline__ void gate_load4(const float* la, int stride, int Lc, int tid, float4 (&g)[8]) {
    const int c4 = tid & 31, rg = tid >> 5;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * rg + i;
        g[i] = r < Lc ? *reinterpret_cast<const float4*>(la + static_cast<size_t>(r) * stride + 4 * c4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

__device__ __forceinline__ float4 add4(const float4& a, const float4& b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d) {
    return make_uint2(pack_bf16(a, b), pack_bf16(c, d));
}

//   g    : this thread's log_alpha rows from gate_load4 (overwritten)
//   opa, opkb, Lc, beta_s, beta_cur, egm/egc/egcm: as gate_chunk; red: f32 [8][128] scratch
//   l2n  : the fused L2 normalisation of the k and q rows, 1 / sqrt(|row|^2 + eps): the warp holds
//          whole rows, so each row's sum of squares is a butterfly over its lanes
__device__ __forceinline__ void gate_chunk4(float4 (&g)[8], uint8_t* opa, uint8_t* opkb, int Lc, float* red,
                                            float* beta_s, float beta_cur, float* egm, float* egc, float* egcm,
                                            int tid, bool l2n = false, float eps = 0.f) {
    const int c4 = tid & 31, rg = tid >> 5;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        acc = add4(acc, g[i]);
        g[i] = acc;
    }
    reinterpret_cast<float4*>(red + rg * D)[c4] = acc;
    if (tid < C) beta_s[tid] = (tid < Lc) ? beta_cur : 0.f;
    __syncthreads();
    float4 off = make_float4(0.f, 0.f, 0.f, 0.f), gm = off, gc = off;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 pq = reinterpret_cast<const float4*>(red + q * D)[c4];
        if (q < rg) off = add4(off, pq);
        if (q < 4) gm = add4(gm, pq);  // g at row 31, the last row of group 3
        gc = add4(gc, pq);
    }
    if (rg == 0) {
        *reinterpret_cast<float4*>(egm + 4 * c4) = make_float4(expf(gm.x), expf(gm.y), expf(gm.z), expf(gm.w));
        *reinterpret_cast<float4*>(egc + 4 * c4) = make_float4(expf(gc.x), expf(gc.y), expf(gc.z), expf(gc.w));
        *reinterpret_cast<float4*>(egcm + 4 * c4) =
            make_float4(expf(gc.x - gm.x), expf(gc.y - gm.y), expf(gc.z - gm.z), expf(gc.w - gm.w));
    }
    const float4 cc = make_float4((off.x - gm.x) * kLog2e, (off.y - gm.y) * kLog2e, (off.z - gm.z) * kLog2e,
                                  (off.w - gm.w) * kLog2e);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * rg + i;
        const float x0 = fmaf(g[i].x, kLog2e, cc.x), x1 = fmaf(g[i].y, kLog2e, cc.y);
        const float x2 = fmaf(g[i].z, kLog2e, cc.z), x3 = fmaf(g[i].w, kLog2e, cc.w);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1), e2 = ex2_approx(x2), e3 = ex2_approx(x3);
        const float f0 = ex2_approx(-x0), f1 = ex2_approx(-x1), f2 = ex2_approx(-x2), f3 = ex2_approx(-x3);
        const uint32_t koff = sw128_off(r, 4 * c4, 16384);
        const uint32_t qoff = sw128_off(64 + r, 4 * c4, 16384);
        float2 k01 = make_float2(0.f, 0.f), k23 = k01, q01 = k01, q23 = k01;
        if (r < Lc) {
            const uint2 kw = *reinterpret_cast<const uint2*>(opa + koff);
            const uint2 qw = *reinterpret_cast<const uint2*>(opa + qoff);
            k01 = unpack_bf16(kw.x); k23 = unpack_bf16(kw.y);
            q01 = unpack_bf16(qw.x); q23 = unpack_bf16(qw.y);
            if (l2n) {  // fused L2 normalisation of k and q rows (r < Lc is uniform over the warp)
                float sk = k01.x * k01.x + k01.y * k01.y + k23.x * k23.x + k23.y * k23.y;
                float sq = q01.x * q01.x + q01.y * q01.y + q23.x * q23.x + q23.y * q23.y;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    sk += __shfl_xor_sync(0xffffffffu, sk, o);
                    sq += __shfl_xor_sync(0xffffffffu, sq, o);
                }
                const float ik = rsqrtf(sk + eps), iq = rsqrtf(sq + eps);
                k01.x *= ik; k01.y *= ik; k23.x *= ik; k23.y *= ik;
                q01.x *= iq; q01.y *= iq; q23.x *= iq; q23.y *= iq;
            }
        }
        *reinterpret_cast<uint2*>(opa + koff) = pack4(k01.x * e0, k01.y * e1, k23.x * e2, k23.y * e3);
        *reinterpret_cast<uint2*>(opa + qoff) = pack4(q01.x * e0, q01.y * e1, q23.x * e2, q23.y * e3);
        *reinterpret_cast<uint2*>(opkb + sw128_off(r, 4 * c4, 8192)) =
            pack4(k01.x * f0, k01.y * f1, k23.x * f2, k23.y * f3);
    }
}

// Write N = Diag(beta) strict_lower(A) for row r (32 columns starting at
// 32*hw) from a 32-column TMEM read into the fp32 scratch.
__device__ __forceinline__ void store_n_row(float* Nf, int r, int hw, float br, const float* a) {
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
        const int i0 = 32 * hw + 4 * j4;
        m4(Nf, r, 8 * hw + j4) =
            make_float4(i0 + 0 < r ? br * a[4 * j4 + 0] : 0.f, i0 + 1 < r ? br * a[4 * j4 + 1] : 0.f,
                        i0 + 2 < r ? br * a[4 * j4 + 2] : 0.f, i0 + 3 < r ? br * a[4 * j4 + 3] : 0.f);
    }
}

// M row rr: lower(Qh Kb^T) entries i <= rr of 32 columns starting at 32*hw,
// as bf16 into a 128B-swizzled row (chunks 4hw..4hw+3).
__device__ __forceinline__ void store_m_row(uint8_t* tile, int row, int rr, int hw, const float* a) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = (32 * hw + 8 * ch + e <= rr) ? a[8 * ch + e] : 0.f;
        *reinterpret_cast<uint4*>(tile + sw128_chunk(row, 4 * hw + ch)) = pack8(m8);
    }
}

// Tb = T Diag(beta) (lower incl. diagonal) -> bf16 rows 0..63 of a swizzled tile.
__device__ __forceinline__ void store_tb(uint8_t* tile, const Rows64& Tf, const float* beta_s, int tid) {
    const int r = tid >> 2, c0 = 16 * (tid & 3);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float m8[8];
#pragma unroll
        for (int e4 = 0; e4 < 2; ++e4) {
            const int i0 = c0 + 8 * hf + 4 * e4;
            const float4 tv = m4(Tf, r, i0 >> 2);
            const float4 bv = *reinterpret_cast<const float4*>(beta_s + i0);
            m8[4 * e4 + 0] = i0 + 0 <= r ? tv.x * bv.x : 0.f;
            m8[4 * e4 + 1] = i0 + 1 <= r ? tv.y * bv.y : 0.f;
            m8[4 * e4 + 2] = i0 + 2 <= r ? tv.z * bv.z : 0.f;
            m8[4 * e4 + 3] = i0 + 3 <= r ? tv.w * bv.w : 0.f;
        }
        *reinterpret_cast<uint4*>(tile + sw128_chunk(r, (c0 >> 3) + hf)) = pack8(m8);
    }
}

// Diagonal 16 x 16 blocks of T = (I + N)^-1 for strictly lower N (64 x 64, fp32) by forward
// substitution (warps 0..3, one column per lane of the first half-warp).  No barrier inside.
__device__ __forceinline__ void lower_inverse_diag_col(const Rows64& Nf, const Rows64& Tf, int B, int j);
__device__ __forceinline__ void lower_inverse_diag(const Rows64& Nf, const Rows64& Tf, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < 4 && lane < 16) lower_inverse_diag_col(Nf, Tf, warp, lane);
}
// Column j of diagonal block B of T by forward substitution (one thread).
__device__ __forceinline__ void lower_inverse_diag_col(const Rows64& Nf, const Rows64& Tf, int B, int j) {
    {
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int row = 16 * B + r;
            float nv[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                if (4 * q4 < r) {
                    const float4 v = m4(Nf, row, 4 * B + q4);
                    nv[4 * q4] = v.x; nv[4 * q4 + 1] = v.y; nv[4 * q4 + 2] = v.z; nv[4 * q4 + 3] = v.w;
                }
            }
            float s0 = (r == j) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i + 1 < r; i += 2) {
                s0 = fmaf(-nv[i], t[i], s0);
                s1 = fmaf(-nv[i + 1], t[i + 1], s1);
            }
            if (r & 1) s0 = fmaf(-nv[r - 1], t[r - 1], s0);
            t[r] = s0 + s1;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) m1(Tf, 16 * B + r, 16 * B + j) = t[r];
    }
}

// T = (I + N)^-1 for strictly lower N (64 x 64, fp32), by 16 x 16 blocks: the diagonal blocks T_II by
// forward substitution (lower_inverse_diag), then, with the block products on the tensor cores,
//   (a) the two 32 x 32 diagonal halves:  T_10 = -T_11 (N_10 T_00),  T_32 = -T_33 (N_32 T_22)
//       (four warps, one 16 x 8 column tile each, X staged through the warp's own slot of Xs);
//   (b) the lower-left 32 x 32 block of the halves T_ll, T_hh just completed:
//       X = N_hl T_ll, then T_hl = -T_hh X  (all eight warps, one 16 x 8 tile of the 32 x 32 result
//       each; X through Xs as [32][40] fp32, a barrier between the two products).
// tf32 mma.sync products with fp32 accumulation; the operands are rounded to tf32 (2^-11), below the
// bf16 rounding Tb takes afterwards.  Only blocks on or below the diagonal are read.  Needs NT >= 256
// threads and 1280 floats of Xs; ends synchronised.  diag_done: the caller has solved the diagonal
// blocks and synchronised.
constexpr int kInvScratchFloats = 32 * 40;
__device__ __forceinline__ void lower_inverse_tc(const Rows64& Nf, const Rows64& Tf, float* Xs, int tid,
                                                 bool diag_done = false) {
    if (!diag_done) {
        lower_inverse_diag(Nf, Tf, tid);
        __syncthreads();
    }
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    if (warp < 4) {  // (a) block (R, I) = (I + 1, I), I = 0 or 2; column tile n0
        const int I = 2 * (warp >> 1), R = I + 1, n0 = 16 * I + 8 * (warp & 1);
        float* xs = Xs + warp * 128;  // [16][8]
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 16; kk += 8) {
            const int k0 = 16 * I + kk;
            const uint32_t a[4] = {to_tf32(m1(Nf, 16 * R + g, k0 + t)), to_tf32(m1(Nf, 16 * R + g + 8, k0 + t)),
                                   to_tf32(m1(Nf, 16 * R + g, k0 + t + 4)),
                                   to_tf32(m1(Nf, 16 * R + g + 8, k0 + t + 4))};
            mma_tf32(x, a, to_tf32(m1(Tf, k0 + t, n0 + g)), to_tf32(m1(Tf, k0 + t + 4, n0 + g)));
        }
        xs[g * 8 + 2 * t] = x[0];
        xs[g * 8 + 2 * t + 1] = x[1];
        xs[(g + 8) * 8 + 2 * t] = x[2];
        xs[(g + 8) * 8 + 2 * t + 1] = x[3];
        __syncwarp();
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 16; kk += 8) {
            const int k0 = 16 * R + kk;
            const uint32_t a[4] = {to_tf32(m1(Tf, 16 * R + g, k0 + t)), to_tf32(m1(Tf, 16 * R + g + 8, k0 + t)),
                                   to_tf32(m1(Tf, 16 * R + g, k0 + t + 4)),
                                   to_tf32(m1(Tf, 16 * R + g + 8, k0 + t + 4))};
            mma_tf32(y, a, to_tf32(xs[(kk + t) * 8 + g]), to_tf32(xs[(kk + t + 4) * 8 + g]));
        }
        // columns n0 + 2t, +1 share one swizzled float4 group: one 8-byte store per row
        *reinterpret_cast<float2*>(&m1(Tf, 16 * R + g, n0 + 2 * t)) = make_float2(-y[0], -y[1]);
        *reinterpret_cast<float2*>(&m1(Tf, 16 * R + g + 8, n0 + 2 * t)) = make_float2(-y[2], -y[3]);
    }
    __syncthreads();
    // (b) warp -> rows 16 rb .. of the 32 x 32 block (rows 32 + 16 rb of T), columns n0 .. n0 + 7
    constexpr int LX = 40;  // Xs row stride: the paired stores and the B reads below hit distinct banks
    const int rb = warp & 1, n0 = 8 * (warp >> 1);
    {   // X = N_hl T_ll; T_ll[k][n] = 0 for k in an upper block, so columns 16.. need k >= 16 only
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        const int r = 32 + 16 * rb;
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8) {
            if (n0 >= 16 && k0 < 16) continue;
            const uint32_t a[4] = {to_tf32(m1(Nf, r + g, k0 + t)), to_tf32(m1(Nf, r + g + 8, k0 + t)),
                                   to_tf32(m1(Nf, r + g, k0 + t + 4)), to_tf32(m1(Nf, r + g + 8, k0 + t + 4))};
            mma_tf32(x, a, to_tf32(m1(Tf, k0 + t, n0 + g)), to_tf32(m1(Tf, k0 + t + 4, n0 + g)));
        }
        *reinterpret_cast<float2*>(Xs + (16 * rb + g) * LX + n0 + 2 * t) = make_float2(x[0], x[1]);
        *reinterpret_cast<float2*>(Xs + (16 * rb + g + 8) * LX + n0 + 2 * t) = make_float2(x[2], x[3]);
    }
    __syncthreads();
    {   // T_hl = -T_hh X; row block rb of T_hh is nonzero in columns 32 .. 32 + 16 rb + 15 only
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        const int r = 32 + 16 * rb;
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8) {
            if (k0 >= 16 * (rb + 1)) continue;
            const uint32_t a[4] = {to_tf32(m1(Tf, r + g, 32 + k0 + t)), to_tf32(m1(Tf, r + g + 8, 32 + k0 + t)),
                                   to_tf32(m1(Tf, r + g, 32 + k0 + t + 4)),
                                   to_tf32(m1(Tf, r + g + 8, 32 + k0 + t + 4))};
            mma_tf32(y, a, to_tf32(Xs[(k0 + t) * LX + n0 + g]), to_tf32(Xs[(k0 + t + 4) * LX + n0 + g]));
        }
        *reinterpret_cast<float2*>(&m1(Tf, r + g, n0 + 2 * t)) = make_float2(-y[0], -y[1]);
        *reinterpret_cast<float2*>(&m1(Tf, r + g + 8, n0 + 2 * t)) = make_float2(-y[2], -y[3]);
    }
    __syncthreads();
}

}  // namespace pf
}  // namespace kda
