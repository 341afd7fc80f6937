// kda_prefill.cu -- chunkwise-parallel KDA prefill on sm_103a (tcgen05 + TMEM + TMA).
//
// "Understanding Kimi Delta Attention" (pyshine), section "The Chunkwise DPLR
// Algorithm": the recurrence is processed in fixed-size chunks as a sequence
// of small matrix operations that stays exactly equivalent to the token loop.
// The pages give no chunk equations; the algebra below is derived from the KDA
// equation (same page, "The KDA Recurrence") and o_t = S_t^T q_t ("kimi delta
// attn from first principles" (aryagxr), section "KDA").
//
// Per chunk of C = 64 rows with start state S (dk x dv, rows = key channels):
//   g   = inclusive cumsum of log_alpha over the chunk rows (per channel)
//   gm  = g at row 31 (reference row), gC = g at row 63
//   Kh  = k*exp(g-gm),  Qh = q*exp(g-gm),  Kb = k*exp(gm-g)            (bf16)
//   A   = Kh Kb^T (strictly lower part),  QK = Qh Kb^T (lower incl. diag)
//   T   = (I + Diag(beta) A)^-1 (fp32 forward substitution), Tb = T Diag(beta)
//   [W; MW]  = [Tb; M Tb] Kh,     [U0; MU0] = [Tb; M Tb] V
//   [U; O]   = [U0; MU0] + [-W; Qh - MW] (Diag(exp(gm)) S)
//   S       <- Diag(exp(gC)) S + Diag(exp(gC-gm)) Kb^T U
// Rows past the sequence end are masked to k = q = v = 0, beta = 0,
// log_alpha = 0, which makes them exact no-ops.
//
// Each CTA owns one (sequence, head) and walks its chunks in order; the state
// stays on chip in registers (fp32) for the whole sequence.  All contractions
// run on the 5th-generation tensor cores: one thread issues tcgen05.mma from
// shared-memory descriptors into TMEM accumulators, and the 256 threads read
// TMEM back with tcgen05.ld for the elementwise steps.  q, k, v and log_alpha
// arrive by TMA (cp.async.bulk.tensor), the next chunk's loads overlapping the
// current chunk's work.  All on-chip waits are bounded; on expiry the kernel
// sets KDA_DEV_TIMEOUT and winds down instead of hanging.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;     // 64
constexpr int D = kHeadDim;   // 128
constexpr int NT = 256;       // threads per CTA
constexpr long long kWaitLimit = 4000000000LL;  // ~2 s of SM clock

// Shared-memory map (bytes from a 1024-aligned base).  NV = dv columns per CTA.
template <int NV>
struct Smem {
    static constexpr uint32_t STAGE_Q = 0;                    // [64][128] bf16, plain rows (TMA)
    static constexpr uint32_t STAGE_K = STAGE_Q + C * D * 2;  // [64][128] bf16
    static constexpr uint32_t STAGE_LA = STAGE_K + C * D * 2; // [64][128] f32
    static constexpr uint32_t OP_A = STAGE_LA + C * D * 4;    // [2 blk][128 rows][128 B]: [Kh;Qh] then [-W; Qh-MW]
    static constexpr uint32_t OP_KB = OP_A + 2 * 128 * 128;   // [2 blk][64 rows][128 B]: Kb
    static constexpr uint32_t OP_A3 = OP_KB + 2 * 64 * 128;   // [1 blk][128 rows][128 B]: [Tb; M] then [Tb; M Tb]
    static constexpr uint32_t OP_V = OP_A3 + 128 * 128;       // [NV/64 blk][64 rows][128 B] (TMA, swizzled)
    static constexpr uint32_t OP_SM = OP_V + (NV / 64) * 64 * 128;   // [NV/64][128 rows][128 B]: bf16 Diag(e^gm) S
    static constexpr uint32_t OP_U = OP_SM + (NV / 64) * 128 * 128;  // [NV/64][64 rows][128 B]: bf16 U
    static constexpr uint32_t END_OPS = OP_U + (NV / 64) * 64 * 128;
    // fp32 scratch of the triangular inverse: N[64][65], T[64][65], X[3][16][16]
    static constexpr uint32_t INV_BYTES = 2 * 64 * 65 * 4 + 3 * 256 * 4;
    static constexpr bool INV_ALIASES_CHAIN = (END_OPS - OP_SM) >= INV_BYTES;
    static constexpr uint32_t INV = INV_ALIASES_CHAIN ? OP_SM : END_OPS;
    static constexpr uint32_t SMALL = INV_ALIASES_CHAIN ? END_OPS : ((END_OPS + INV_BYTES + 1023) / 1024) * 1024;
    // small region
    static constexpr uint32_t BETA = SMALL;                 // f32[64]
    static constexpr uint32_t RED = BETA + 64 * 4;          // f32[4][128] cumsum partials
    static constexpr uint32_t EGM = RED + 4 * 128 * 4;      // f32[128] exp(gm)
    static constexpr uint32_t EGC = EGM + 128 * 4;          // f32[128] exp(gC)
    static constexpr uint32_t EGCM = EGC + 128 * 4;         // f32[128] exp(gC - gm)
    static constexpr uint32_t BARS = EGCM + 128 * 4;        // 3 x u64 mbarriers
    static constexpr uint32_t TMEM_SLOT = BARS + 3 * 8;     // u32
    static constexpr uint32_t ABORT = TMEM_SLOT + 4;        // i32
    static constexpr uint32_t TOTAL = ABORT + 4;
    static constexpr uint32_t ALLOC = TOTAL + 1024;         // + alignment slack
};

// TMEM column map (512 columns allocated).
constexpr uint32_t TM_D1 = 0;    // 64 cols: [A; QK], later [*; M Tb]
constexpr uint32_t TM_D3 = 64;   // 128 cols: [W; MW]
constexpr uint32_t TM_X = 192;   // NV cols: [U0; MU0] + [-W; Qh-MW] Sm = [U; O]
// TM_S = TM_X + NV: Kb^T U

__device__ __forceinline__ uint32_t tmem_lane(int quarter) { return static_cast<uint32_t>(32 * quarter) << 16; }

template <typename OutT>
__device__ __forceinline__ void store_out8(OutT* dst, const float* v);
template <>
__device__ __forceinline__ void store_out8<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
    uint4 pk;
    pk.x = pack_bf16(v[0], v[1]);
    pk.y = pack_bf16(v[2], v[3]);
    pk.z = pack_bf16(v[4], v[5]);
    pk.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = pk;
}
template <>
__device__ __forceinline__ void store_out8<float>(float* dst, const float* v) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

template <int NV, typename OutT>
__global__ void __launch_bounds__(NT, 1)
    kda_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
                       const PrefillArgs p) {
    using L = Smem<NV>;
    constexpr int NSLICE = D / NV;
    constexpr int SC = NV / 2;  // state columns per thread
    static_assert(NV == 128 || NV == 64, "dv slice must be 64 or 128");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qw = warp & 3;   // TMEM lane quarter this warp may access
    const int hw = warp >> 2;  // column half
    const int H = p.H;

    const int unit = blockIdx.x;
    const int slice = unit % NSLICE;
    const int h = (unit / NSLICE) % H;
    const int pos = unit / (NSLICE * H);
    const int seq = p.order ? p.order[pos] : pos;
    const int j0 = slice * NV;

    const int64_t t_begin = p.cu_seqlens[seq];
    const int64_t t_end = p.cu_seqlens[seq + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.total_tokens) {
        if (tid == 0 && p.device_status) atomicOr(p.device_status, KDA_DEV_BAD_CU_SEQLENS);
        return;
    }
    const int nch = static_cast<int>((t_end - t_begin + C - 1) / C);

    // ---- state: row rho of S, columns [j0 + hw*SC, +SC) in registers ----
    const int rho = 32 * qw + lane;
    float S[SC];
    const size_t srow = ((static_cast<size_t>(seq) * H + h) * D + rho) * D + j0 + hw * SC;
    if (p.S0) {
#pragma unroll
        for (int j = 0; j < SC; j += 4) {
            const float4 t = *reinterpret_cast<const float4*>(p.S0 + srow + j);
            S[j] = t.x; S[j + 1] = t.y; S[j + 2] = t.z; S[j + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < SC; ++j) S[j] = 0.f;
    }
    if (nch == 0) {
        if (p.S_final) {
#pragma unroll
            for (int j = 0; j < SC; j += 4)
                *reinterpret_cast<float4*>(p.S_final + srow + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
        return;
    }

    uint64_t* bar_in = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_v = bar_in + 1;
    uint64_t* bar_mma = bar_in + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::TMEM_SLOT);
    volatile int* abort_s = reinterpret_cast<volatile int*>(sm + L::ABORT);
    float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
    float* red = reinterpret_cast<float*>(sm + L::RED);
    float* egm = reinterpret_cast<float*>(sm + L::EGM);
    float* egc = reinterpret_cast<float*>(sm + L::EGC);
    float* egcm = reinterpret_cast<float*>(sm + L::EGCM);
    float* Nf = reinterpret_cast<float*>(sm + L::INV);
    float* Tf = Nf + 64 * 65;
    float* Xs = Tf + 64 * 65;

    if (tid == 0) {
        mbar_init(bar_in, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        *abort_s = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_la);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_q = tmem + tmem_lane(qw);  // this warp's lane quarter
    constexpr uint32_t TM_S = TM_X + NV;

    constexpr uint32_t kInBytes = C * D * 2 * 2 + C * D * 4;  // q + k + log_alpha
    constexpr uint32_t kVBytes = (NV / 64) * 64 * 128;

    auto issue_in = [&](int c) {
        const int32_t t0 = static_cast<int32_t>(t_begin + static_cast<int64_t>(c) * C);
        mbar_arrive_expect_tx(bar_in, kInBytes);
        tma_load_3d(sm + L::STAGE_Q, &tm_q, bar_in, 0, h, t0);
        tma_load_3d(sm + L::STAGE_K, &tm_k, bar_in, 0, h, t0);
        tma_load_3d(sm + L::STAGE_LA, &tm_la, bar_in, 0, h, t0);
    };
    auto issue_v = [&](int c) {
        const int32_t t0 = static_cast<int32_t>(t_begin + static_cast<int64_t>(c) * C);
        mbar_arrive_expect_tx(bar_v, kVBytes);
#pragma unroll
        for (int b = 0; b < NV / 64; ++b) tma_load_3d(sm + L::OP_V + b * 8192, &tm_v, bar_v, j0 + 64 * b, h, t0);
    };

    bool in_flight_in = false, in_flight_v = false;  // meaningful on thread 0 only
    if (tid == 0) {
        issue_in(0);
        issue_v(0);
        in_flight_in = in_flight_v = true;
    }
    // beta of the next chunk is prefetched into a register by threads 0..63
    float beta_next = 0.f;
    if (tid < C && tid < t_end - t_begin) beta_next = p.beta[(t_begin + tid) * H + h];

    uint32_t ph_in = 0, ph_v = 0, ph_mma = 0;
    auto wait_or_abort = [&](uint64_t* bar, uint32_t& ph) {
        if (!mbar_wait(bar, ph, kWaitLimit)) {
            *abort_s = 1;
            if (p.device_status) atomicOr(p.device_status, KDA_DEV_TIMEOUT);
        }
        ph ^= 1u;
    };
    auto mma_round = [&]() {  // all threads: wait for the last commit, then order TMEM reads after it
        wait_or_abort(bar_mma, ph_mma);
        tc_fence_after();
    };

    const uint32_t a_base = smem_u32(sm + L::OP_A);
    const uint32_t kb_base = smem_u32(sm + L::OP_KB);
    const uint32_t a3_base = smem_u32(sm + L::OP_A3);
    const uint32_t v_base = smem_u32(sm + L::OP_V);
    const uint32_t sm_base = smem_u32(sm + L::OP_SM);
    const uint32_t u_base = smem_u32(sm + L::OP_U);

    for (int c = 0; c < nch; ++c) {
        const int64_t t0 = t_begin + static_cast<int64_t>(c) * C;
        const int Lc = static_cast<int>(t_end - t0 < C ? t_end - t0 : C);

        // ================= step E: gates, gated operands =================
        if (tid == 0) in_flight_in = false;
        wait_or_abort(bar_in, ph_in);
        {
            const int cp = tid & 63;  // channel pair (2cp, 2cp+1)
            const int rq = tid >> 6;  // rows 16rq .. 16rq+15
            const float* la_s = reinterpret_cast<const float*>(sm + L::STAGE_LA);
            float g0[16], g1[16];
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * rq + i;
                float2 l2 = make_float2(0.f, 0.f);
                if (r < Lc) l2 = *reinterpret_cast<const float2*>(la_s + r * D + 2 * cp);
                acc0 += l2.x;
                acc1 += l2.y;
                g0[i] = acc0;
                g1[i] = acc1;
            }
            reinterpret_cast<float2*>(red + rq * D)[cp] = make_float2(acc0, acc1);
            if (tid < C) beta_s[tid] = (tid < Lc) ? beta_next : 0.f;
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
            const uint32_t* qs = reinterpret_cast<const uint32_t*>(sm + L::STAGE_Q);
            const uint32_t* ks = reinterpret_cast<const uint32_t*>(sm + L::STAGE_K);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * rq + i;
                const float d0 = g0[i] + off0 - gm0, d1 = g1[i] + off1 - gm1;
                const float e0 = expf(d0), e1 = expf(d1);
                const float f0 = expf(-d0), f1 = expf(-d1);
                float2 kk = make_float2(0.f, 0.f), qv = kk;
                if (r < Lc) {
                    kk = unpack_bf16(ks[r * 64 + cp]);
                    qv = unpack_bf16(qs[r * 64 + cp]);
                }
                *reinterpret_cast<uint32_t*>(sm + L::OP_A + sw128_off(r, 2 * cp, 16384)) =
                    pack_bf16(kk.x * e0, kk.y * e1);
                *reinterpret_cast<uint32_t*>(sm + L::OP_A + sw128_off(64 + r, 2 * cp, 16384)) =
                    pack_bf16(qv.x * e0, qv.y * e1);
                *reinterpret_cast<uint32_t*>(sm + L::OP_KB + sw128_off(r, 2 * cp, 8192)) =
                    pack_bf16(kk.x * f0, kk.y * f1);
            }
        }
        // V of this chunk: wait for its TMA; zero rows past the sequence end
        if (tid == 0) in_flight_v = false;
        wait_or_abort(bar_v, ph_v);
        if (Lc < C) {
            const int nz = (C - Lc) * (NV / 8);  // 16-byte chunks to clear
            for (int e = tid; e < nz; e += NT) {
                const int r = Lc + e / (NV / 8), ch = e % (NV / 8);
                *reinterpret_cast<uint4*>(sm + L::OP_V + (ch >> 3) * 8192 + sw128_chunk(r, ch & 7)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        // next chunk's beta
        if (tid < C) {
            beta_next = 0.f;
            if (c + 1 < nch && t0 + C + tid < t_end) beta_next = p.beta[(t0 + C + tid) * H + h];
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*abort_s) break;

        // ================= MMA1: [Kh; Qh] Kb^T -> D1 (128 x 64) =================
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t koff = (s >> 2) * 16384 + (s & 3) * 32;
                const uint32_t kboff = (s >> 2) * 8192 + (s & 3) * 32;
                mma_bf16(tmem + TM_D1, sdesc_sw128(a_base + koff, 16, 1024), sdesc_sw128(kb_base + kboff, 16, 1024),
                         id, s > 0);
            }
            mma_commit(bar_mma);
            // staging is free: prefetch the next chunk's q, k, log_alpha
            if (c + 1 < nch) {
                fence_async_smem();
                issue_in(c + 1);
                in_flight_in = true;
            }
        }
        mma_round();

        // ---- D1 readout: N = Diag(beta) strict_lower(A) (fp32 smem), M = lower(QK) (bf16 operand) ----
        {
            float a[32];
            tmem_ld32(tmem_q + TM_D1 + 32 * hw, a);
            tmem_ld_wait();
            if (qw < 2) {
                const int r = 32 * qw + lane;
                const float br = beta_s[r];
                float* Nrow = Nf + r * 65;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int i = 32 * hw + j;
                    Nrow[i] = (i < r) ? br * a[j] : 0.f;
                }
            } else {
                const int rr = 32 * (qw - 2) + lane;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    float m8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 32 * hw + 8 * ch + e;
                        m8[e] = (i <= rr) ? a[8 * ch + e] : 0.f;
                    }
                    uint4 pk;
                    pk.x = pack_bf16(m8[0], m8[1]);
                    pk.y = pack_bf16(m8[2], m8[3]);
                    pk.z = pack_bf16(m8[4], m8[5]);
                    pk.w = pack_bf16(m8[6], m8[7]);
                    *reinterpret_cast<uint4*>(sm + L::OP_A3 + sw128_chunk(64 + rr, 4 * hw + ch)) = pk;
                }
            }
        }
        tc_fence_before();
        __syncthreads();

        // ---- T = (I + N)^-1: 16x16 diagonal blocks by forward substitution ----
        if (warp < 4 && lane < 16) {
            const int B = warp, j = lane;
            float t[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float* Nr = Nf + (16 * B + r) * 65 + 16 * B;
                float s0 = (r == j) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
                for (int i = 0; i + 1 < r; i += 2) {
                    s0 = fmaf(-Nr[i], t[i], s0);
                    s1 = fmaf(-Nr[i + 1], t[i + 1], s1);
                }
                if (r & 1) s0 = fmaf(-Nr[r - 1], t[r - 1], s0);
                t[r] = s0 + s1;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tf[(16 * B + r) * 65 + 16 * B + j] = t[r];
        }
        __syncthreads();
        // ---- off-diagonal blocks, by distance d = R - I:
        //      T_RI = -T_RR * sum_{J=I}^{R-1} N_RJ T_JI ----
#pragma unroll 1
        for (int d = 1; d <= 3; ++d) {
            const int nout = (4 - d) * 256;
            for (int e = tid; e < nout; e += NT) {
                const int I = e >> 8, r = (e >> 4) & 15, cc = e & 15, R = I + d;
                float s = 0.f;
                for (int J = I; J < R; ++J) {
                    const float* Nr = Nf + (16 * R + r) * 65 + 16 * J;
                    const float* Tc = Tf + (16 * J) * 65 + 16 * I + cc;
#pragma unroll
                    for (int m = 0; m < 16; ++m) s = fmaf(Nr[m], Tc[m * 65], s);
                }
                Xs[e] = s;
            }
            __syncthreads();
            for (int e = tid; e < nout; e += NT) {
                const int I = e >> 8, r = (e >> 4) & 15, cc = e & 15, R = I + d;
                const float* Tr = Tf + (16 * R + r) * 65 + 16 * R;
                const float* Xc = Xs + (I << 8) + cc;
                float s = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m) s = fmaf(Tr[m], Xc[m * 16], s);
                Tf[(16 * R + r) * 65 + 16 * I + cc] = -s;
            }
            __syncthreads();
        }
        // ---- Tb = T Diag(beta) -> bf16 rows 0..63 of OP_A3 ----
        {
            const int r = tid >> 2, c0 = 16 * (tid & 3);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = c0 + 8 * hf + e;
                    m8[e] = (i <= r) ? Tf[r * 65 + i] * beta_s[i] : 0.f;
                }
                uint4 pk;
                pk.x = pack_bf16(m8[0], m8[1]);
                pk.y = pack_bf16(m8[2], m8[3]);
                pk.z = pack_bf16(m8[4], m8[5]);
                pk.w = pack_bf16(m8[6], m8[7]);
                *reinterpret_cast<uint4*>(sm + L::OP_A3 + sw128_chunk(r, (c0 >> 3) + hf)) = pk;
            }
        }
        fence_async_smem();
        __syncthreads();

        // ================= MMA2: [Tb; M] Tb -> D1 (rows 64..127 = M Tb) =================
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, 64, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + TM_D1, sdesc_sw128(a3_base + s * 32, 16, 1024),
                         sdesc_sw128(a3_base + s * 2048, 8192, 1024), id, s > 0);
            mma_commit(bar_mma);
        }
        mma_round();
        if (qw >= 2) {
            const int rr = 32 * (qw - 2) + lane;
            float a[32];
            tmem_ld32(tmem_q + TM_D1 + 32 * hw, a);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint4 pk;
                pk.x = pack_bf16(a[8 * ch + 0], a[8 * ch + 1]);
                pk.y = pack_bf16(a[8 * ch + 2], a[8 * ch + 3]);
                pk.z = pack_bf16(a[8 * ch + 4], a[8 * ch + 5]);
                pk.w = pack_bf16(a[8 * ch + 6], a[8 * ch + 7]);
                *reinterpret_cast<uint4*>(sm + L::OP_A3 + sw128_chunk(64 + rr, 4 * hw + ch)) = pk;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ================= MMA3: [Tb; M Tb] [Kh | V] -> D3 = [W; MW], X = [U0; MU0] =================
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_w = idesc_bf16_f32(128, 128, false, true);
            constexpr uint32_t id_v = idesc_bf16_f32(128, NV, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + TM_D3, sdesc_sw128(a3_base + s * 32, 16, 1024),
                         sdesc_sw128(a_base + s * 2048, 16384, 1024), id_w, s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + TM_X, sdesc_sw128(a3_base + s * 32, 16, 1024),
                         sdesc_sw128(v_base + s * 2048, 8192, 1024), id_v, s > 0);
            mma_commit(bar_mma);
        }
        mma_round();
        if (tid == 0 && c + 1 < nch) {  // V operand consumed: prefetch the next chunk's V
            issue_v(c + 1);
            in_flight_v = true;
        }
        // ---- A_chain = [-W; Qh - MW] (bf16, K-major, in place of [Kh; Qh]) ----
        {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float a[32];
                tmem_ld32(tmem_q + TM_D3 + 64 * hw + 32 * half, a);
                tmem_ld_wait();
                const int row = 32 * qw + lane;  // 0..127 of the stacked operand
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const int chunk = 4 * half + ch;  // 16-byte chunk within column block hw
                    uint8_t* dst = sm + L::OP_A + hw * 16384 + sw128_chunk(row, chunk);
                    float m8[8];
                    if (qw < 2) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) m8[e] = -a[8 * ch + e];
                    } else {
                        const uint4 old = *reinterpret_cast<const uint4*>(dst);
                        const float2 q0 = unpack_bf16(old.x), q1 = unpack_bf16(old.y);
                        const float2 q2 = unpack_bf16(old.z), q3 = unpack_bf16(old.w);
                        m8[0] = q0.x - a[8 * ch + 0]; m8[1] = q0.y - a[8 * ch + 1];
                        m8[2] = q1.x - a[8 * ch + 2]; m8[3] = q1.y - a[8 * ch + 3];
                        m8[4] = q2.x - a[8 * ch + 4]; m8[5] = q2.y - a[8 * ch + 5];
                        m8[6] = q3.x - a[8 * ch + 6]; m8[7] = q3.y - a[8 * ch + 7];
                    }
                    uint4 pk;
                    pk.x = pack_bf16(m8[0], m8[1]);
                    pk.y = pack_bf16(m8[2], m8[3]);
                    pk.z = pack_bf16(m8[4], m8[5]);
                    pk.w = pack_bf16(m8[6], m8[7]);
                    *reinterpret_cast<uint4*>(dst) = pk;
                }
            }
        }
        // ---- Sm = Diag(exp(gm)) S -> bf16 MN-major operand (row rho, this thread's columns) ----
        {
            const float sc = egm[rho];
#pragma unroll
            for (int ch = 0; ch < SC / 8; ++ch) {
                const int col = hw * SC + 8 * ch;  // column within the slice
                uint4 pk;
                pk.x = pack_bf16(sc * S[8 * ch + 0], sc * S[8 * ch + 1]);
                pk.y = pack_bf16(sc * S[8 * ch + 2], sc * S[8 * ch + 3]);
                pk.z = pack_bf16(sc * S[8 * ch + 4], sc * S[8 * ch + 5]);
                pk.w = pack_bf16(sc * S[8 * ch + 6], sc * S[8 * ch + 7]);
                *reinterpret_cast<uint4*>(sm + L::OP_SM + (col >> 6) * 16384 + sw128_chunk(rho, (col & 63) >> 3)) =
                    pk;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ================= chain MMA1: X += A_chain Sm  ->  [U; O] =================
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, NV, false, true);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem + TM_X, sdesc_sw128(a_base + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                         sdesc_sw128(sm_base + s * 2048, 16384, 1024), id, 1u);
            mma_commit(bar_mma);
        }
        mma_round();
        // ---- U -> bf16 operand; O -> global ----
        {
#pragma unroll
            for (int part = 0; part < SC / 32; ++part) {
                float a[32];
                tmem_ld32(tmem_q + TM_X + hw * SC + 32 * part, a);
                tmem_ld_wait();
                const int col = hw * SC + 32 * part;  // within the slice
                if (qw < 2) {
                    const int r = 32 * qw + lane;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint4 pk;
                        pk.x = pack_bf16(a[8 * ch + 0], a[8 * ch + 1]);
                        pk.y = pack_bf16(a[8 * ch + 2], a[8 * ch + 3]);
                        pk.z = pack_bf16(a[8 * ch + 4], a[8 * ch + 5]);
                        pk.w = pack_bf16(a[8 * ch + 6], a[8 * ch + 7]);
                        const int cc = col + 8 * ch;
                        *reinterpret_cast<uint4*>(sm + L::OP_U + (cc >> 6) * 8192 + sw128_chunk(r, (cc & 63) >> 3)) =
                            pk;
                    }
                } else {
                    const int rr = 32 * (qw - 2) + lane;
                    if (rr < Lc) {
                        OutT* dst = static_cast<OutT*>(p.o) + ((t0 + rr) * H + h) * static_cast<int64_t>(D) + j0 + col;
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) store_out8<OutT>(dst + 8 * ch, a + 8 * ch);
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ================= chain MMA2: Kb^T U -> TM_S (128 x NV) =================
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, NV, true, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + TM_S, sdesc_sw128(kb_base + s * 2048, 8192, 1024),
                         sdesc_sw128(u_base + s * 2048, 8192, 1024), id, s > 0);
            mma_commit(bar_mma);
        }
        mma_round();
        // ---- S <- Diag(exp(gC)) S + Diag(exp(gC - gm)) Kb^T U ----
        {
            const float dc = egc[rho], dcm = egcm[rho];
#pragma unroll
            for (int part = 0; part < SC / 32; ++part) {
                float a[32];
                tmem_ld32(tmem_q + TM_S + hw * SC + 32 * part, a);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) S[32 * part + j] = fmaf(dc, S[32 * part + j], dcm * a[j]);
            }
        }
        tc_fence_before();
        // the next iteration's first __syncthreads orders these TMEM reads
        // before any later MMA
    }

    __syncthreads();
    const bool aborted = *abort_s != 0;
    if (tid == 0 && aborted) {  // let any TMA still in flight land before the CTA exits
        if (in_flight_in) (void)mbar_wait(bar_in, ph_in, kWaitLimit);
        if (in_flight_v) (void)mbar_wait(bar_v, ph_v, kWaitLimit);
    }
    if (p.S_final && !aborted) {
#pragma unroll
        for (int j = 0; j < SC; j += 4)
            *reinterpret_cast<float4*>(p.S_final + srow + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------
__global__ void kda_schedule_kernel(const int32_t* __restrict__ cu, int32_t N, int64_t total, int32_t* order,
                                    int32_t* device_status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0 && device_status && (cu[0] != 0 || static_cast<int64_t>(cu[N]) != total))
        atomicOr(device_status, KDA_DEV_BAD_CU_SEQLENS);
    if (i >= N) return;
    const int64_t li = static_cast<int64_t>(cu[i + 1]) - cu[i];
    if (li < 0 && device_status) atomicOr(device_status, KDA_DEV_BAD_CU_SEQLENS);
    int rank = 0;  // longest first; ties by index
    for (int j = 0; j < N; ++j) {
        const int64_t lj = static_cast<int64_t>(cu[j + 1]) - cu[j];
        rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
}

__global__ void kda_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, size_t n) {
    const size_t n4 = n / 4;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(src)[i];
        uint2 pk;
        pk.x = pack_bf16(v.x, v.y);
        pk.y = pack_bf16(v.z, v.w);
        reinterpret_cast<uint2*>(dst)[i] = pk;
    }
    const size_t tail = n4 * 4 + blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    if (blockIdx.x == 0 && tail < n) dst[tail] = __float2bfloat16_rn(src[tail]);
}

template <int NV, typename OutT>
cudaError_t launch_prefill_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_la, const PrefillArgs& a, cudaStream_t stream) {
    using L = Smem<NV>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(kda_prefill_kernel<NV, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(L::ALLOC));
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const long long units = static_cast<long long>(a.num_seqs) * a.H * (D / NV);
    if (units == 0) return cudaSuccess;
    kda_prefill_kernel<NV, OutT><<<static_cast<unsigned>(units), NT, L::ALLOC, stream>>>(tm_q, tm_k, tm_v, tm_la, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_schedule(const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t* order,
                            int32_t* device_status, cudaStream_t stream) {
    const int threads = 256;
    const int blocks = num_seqs > 0 ? (num_seqs + threads - 1) / threads : 1;
    kda_schedule_kernel<<<blocks, threads, 0, stream>>>(cu_seqlens, num_seqs, total_tokens, order, device_status);
    return cudaGetLastError();
}

cudaError_t launch_to_bf16(const float* src, void* dst, size_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const size_t n4 = (n + 3) / 4;
    const unsigned blocks = static_cast<unsigned>((n4 + 255) / 256 < 152 * 32 ? (n4 + 255) / 256 : 152 * 32);
    kda_to_bf16_kernel<<<blocks, 256, 0, stream>>>(src, static_cast<__nv_bfloat16*>(dst), n);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_la, const PrefillArgs& a, bool out_f32, cudaStream_t stream) {
    if (out_f32) return launch_prefill_t<128, float>(tm_q, tm_k, tm_v, tm_la, a, stream);
    return launch_prefill_t<128, __nv_bfloat16>(tm_q, tm_k, tm_v, tm_la, a, stream);
}

}  // namespace kda
