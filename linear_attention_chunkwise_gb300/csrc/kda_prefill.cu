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
//   A   = Kh Kb^T (strictly lower part),  M = lower(Qh Kb^T) (incl. diagonal)
//   T   = (I + Diag(beta) A)^-1 (fp32, blocked forward substitution)
//   Tb  = T Diag(beta)
//   W   = Tb Kh,  U0 = Tb V
//   Sm  = Diag(exp(gm)) S                                              (bf16)
//   U   = U0 - W Sm
//   O   = Qh Sm + M U                                  (rows of this chunk's o)
//   S  <- Diag(exp(gC)) S + Diag(exp(gC-gm)) Kb^T U
// Rows past the sequence end are masked to k = q = v = 0, beta = 0,
// log_alpha = 0, which makes them exact no-ops.
//
// Tensor-core mapping (all tcgen05.mma, M = 128, bf16 in, fp32 TMEM out):
//   MMA1:  [A; QhKb^T]  = [Kh; Qh] Kb^T
//   MMA3:  [W; 0]       = [Tb; 0] Kh        and  X = [U0; 0] = [Tb; 0] V
//   CH1:   X          += [-W; Qh] Sm        ->  X = [U; Qh Sm]
//   CH2:   D_S         = Kb^T U             and  X += [0; M] U  ->  X = [U; O]
// so U and O come out of one accumulator tile and M U needs no extra pass.
//
// Schedule.  One CTA owns one (sequence, head) and walks its chunks in order;
// the fp32 state stays in registers.  The sequential part (CH1, CH2 and the
// state update) of chunk c-1 is software-pipelined against the independent
// preparation of chunk c: while the tensor cores run CH1/CH2 of c-1, the CUDA
// cores compute the gates of c and its triangular inverse, and vice versa.
// Operands that both halves touch are double-buffered (by chunk parity) in
// shared memory and TMEM.  q and k arrive by TMA already in the swizzled
// operand layout and are gated in place; log_alpha and v arrive by TMA too,
// one chunk ahead.  All on-chip waits are bounded: on expiry the kernel sets
// KDA_DEV_TIMEOUT and winds down instead of hanging.
#include <cuda_bf16.h>

#include "kda_prefill_common.cuh"

namespace kda {
namespace {

using namespace pf;

// Shared-memory map (bytes from a 1024-aligned base).  Operand tiles use the
// 128B-swizzled layout of kda_ptx.cuh.
struct Smem {
    static constexpr uint32_t LA = 0;                   // [64][128] f32 log_alpha (TMA, plain rows)
    static constexpr uint32_t OP_A = 32768;             // 2 x [2 blk][128 rows][128 B]: [k;q] -> [Kh;Qh] -> [-W;Qh]
    static constexpr uint32_t OP_A_STRIDE = 32768;
    static constexpr uint32_t OP_KB = OP_A + 2 * 32768;  // 2 x [2 blk][64 rows][128 B]: Kb
    static constexpr uint32_t OP_KB_STRIDE = 16384;
    static constexpr uint32_t OP_A3 = OP_KB + 2 * 16384;  // [Tb (64 rows) | zeros (64) | M (64)] x 128 B
    static constexpr uint32_t OP_V = OP_A3 + 3 * 8192;    // [2 blk][64 rows][128 B]: V (TMA, swizzled)
    static constexpr uint32_t OP_SM = OP_V + 16384;       // [2 blk][128 rows][128 B]: Sm
    static constexpr uint32_t INV_N = OP_SM;              // f32 [64][64] (xor-swizzled), aliases OP_SM
    static constexpr uint32_t INV_T = OP_SM + 16384;      // f32 [64][64]
    static constexpr uint32_t OP_U = OP_SM + 32768;       // [2 blk][64 rows][128 B]: U
    static constexpr uint32_t SMALL = OP_U + 16384;
    static constexpr uint32_t XS = SMALL;                 // f32 inverse scratch
    static constexpr uint32_t BETA = XS + kInvScratchFloats * 4;  // f32 [64]
    static constexpr uint32_t RED = BETA + 64 * 4;        // f32 [4][128] cumsum partials
    static constexpr uint32_t EGM = RED + 4 * 128 * 4;    // f32 [128] exp(gm)
    static constexpr uint32_t EGC = EGM + 128 * 4;        // f32 [2][128] exp(gC), by chunk parity
    static constexpr uint32_t EGCM = EGC + 2 * 128 * 4;   // f32 [2][128] exp(gC - gm), by chunk parity
    static constexpr uint32_t BARS = EGCM + 2 * 128 * 4;  // 8 x u64 mbarriers
    static constexpr uint32_t TMEM_SLOT = BARS + 8 * 8;   // u32
    static constexpr uint32_t ABORT = TMEM_SLOT + 4;      // i32
    static constexpr uint32_t TOTAL = ABORT + 4;
    static constexpr uint32_t ALLOC = TOTAL + 1024;       // + alignment slack
};
static_assert(Smem::ALLOC <= 232448, "shared memory over the sm_103 per-CTA limit");

// TMEM columns (512 allocated): D1 / D3 share [0,128); X by chunk parity; D_S.
constexpr uint32_t TM_D = 0;
constexpr uint32_t TM_X0 = 128;
constexpr uint32_t TM_S = 384;

enum Bar { BAR_LA = 0, BAR_QK, BAR_V, BAR_P1, BAR_P3, BAR_C1, BAR_C2, BAR_FIN };

template <typename OutT>
__global__ void __launch_bounds__(NT, 1)
    kda_prefill_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
                       const PrefillArgs p) {
    using L = Smem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qw = warp & 3;   // TMEM lane quarter this warp may access
    const int hw = warp >> 2;  // column half
    const int H = p.H;

    const int pos = blockIdx.x / H;
    const int h = blockIdx.x - pos * H;
    const int seq = p.order ? p.order[pos] : pos;
    if (!KDA_BOUNDS(pos < p.num_seqs && seq >= 0 && seq < p.num_seqs, p.device_status)) return;

    const int64_t t_begin = p.cu_seqlens[seq];
    const int64_t t_end = p.cu_seqlens[seq + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.total_tokens) {
        if (tid == 0 && p.device_status) atomicOr(p.device_status, KDA_DEV_BAD_CU_SEQLENS);
        return;
    }
    const int nch = static_cast<int>((t_end - t_begin + C - 1) / C);

    // ---- state: row rho of S, columns [hw*64, hw*64 + 64) in registers ----
    const int rho = 32 * qw + lane;
    float S[64];
    const size_t srow = ((static_cast<size_t>(seq) * H + h) * D + rho) * D + hw * 64;
    if (p.S0) {
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
            const float4 t = *reinterpret_cast<const float4*>(p.S0 + srow + j);
            S[j] = t.x; S[j + 1] = t.y; S[j + 2] = t.z; S[j + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) S[j] = 0.f;
    }
    if (nch == 0) {
        if (p.S_final) {
#pragma unroll
            for (int j = 0; j < 64; j += 4)
                *reinterpret_cast<float4*>(p.S_final + srow + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
        return;
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::TMEM_SLOT);
    volatile int* abort_s = reinterpret_cast<volatile int*>(sm + L::ABORT);
    float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
    float* red = reinterpret_cast<float*>(sm + L::RED);
    float* egm = reinterpret_cast<float*>(sm + L::EGM);
    float* egc = reinterpret_cast<float*>(sm + L::EGC);
    float* egcm = reinterpret_cast<float*>(sm + L::EGCM);
    float* Nf = reinterpret_cast<float*>(sm + L::INV_N);
    float* Tf = reinterpret_cast<float*>(sm + L::INV_T);
    float* Xs = reinterpret_cast<float*>(sm + L::XS);

    if (tid == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(&bars[i], 1);
        *abort_s = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_la);
    }
    // zero block of OP_A3 (rows 64..127): the [Tb; 0] and [0; M] operands
    for (int e = tid; e < 8192 / 16; e += NT)
        reinterpret_cast<uint4*>(sm + L::OP_A3 + 8192)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tq = tmem + tmem_lane(qw);  // this warp's lane quarter

    auto chunk_t0 = [&](int c) { return static_cast<int32_t>(t_begin + static_cast<int64_t>(c) * C); };
    auto issue_la = [&](int c) {
        mbar_arrive_expect_tx(&bars[BAR_LA], C * D * 4);
        tma_load_3d(sm + L::LA, &tm_la, &bars[BAR_LA], 0, h, chunk_t0(c));
    };
    auto issue_qk = [&](int c) {  // k -> rows 0..63, q -> rows 64..127 of OP_A[c & 1], per 64-channel block
        uint8_t* dst = sm + L::OP_A + (c & 1) * L::OP_A_STRIDE;
        mbar_arrive_expect_tx(&bars[BAR_QK], 4 * 8192);
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
            tma_load_3d(dst + kh * 16384, &tm_k, &bars[BAR_QK], 64 * kh, h, chunk_t0(c));
            tma_load_3d(dst + kh * 16384 + 8192, &tm_q, &bars[BAR_QK], 64 * kh, h, chunk_t0(c));
        }
    };
    auto issue_v = [&](int c) {
        mbar_arrive_expect_tx(&bars[BAR_V], 2 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) tma_load_3d(sm + L::OP_V + b * 8192, &tm_v, &bars[BAR_V], 64 * b, h, chunk_t0(c));
    };

    // in-flight TMA bookkeeping (thread 0 only), for a clean exit after a timeout
    bool fl_la = false, fl_qk = false, fl_v = false;
    if (tid == 0) {
        issue_la(0);
        issue_qk(0);
        issue_v(0);
        fl_la = fl_qk = fl_v = true;
    }
    float beta_next = 0.f;  // beta of the next chunk, prefetched by threads 0..63
    if (tid < C && tid < t_end - t_begin) beta_next = p.beta[(t_begin + tid) * H + h];

    uint32_t ph[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    auto wait_bar = [&](int i) {  // on expiry the phase is waited for again (drain) before going on
        if (!mbar_wait_pipe(&bars[i], ph[i])) {
            *abort_s = 1;
            if (p.device_status) atomicOr(p.device_status, KDA_DEV_TIMEOUT);
        }
        ph[i] ^= 1u;
    };

    const uint32_t a3_base = smem_u32(sm + L::OP_A3);
    const uint32_t v_base = smem_u32(sm + L::OP_V);
    const uint32_t sm_base = smem_u32(sm + L::OP_SM);
    const uint32_t u_base = smem_u32(sm + L::OP_U);
    float mq[32];  // this thread's 32 entries of Qh Kb^T (lanes 64..127), carried across the inverse
    int Lprev = 0;

    for (int c = 0; c <= nch; ++c) {
        const bool P = c < nch;  // prepare chunk c
        const bool Q = c > 0;    // finish chunk c-1 (the sequential part)
        const int b = c & 1, bp = b ^ 1;
        const int Lc = P ? static_cast<int>(t_end - t_begin - static_cast<int64_t>(c) * C < C
                                                ? t_end - t_begin - static_cast<int64_t>(c) * C
                                                : C)
                         : 0;
        uint8_t* opa = sm + L::OP_A + b * L::OP_A_STRIDE;
        uint8_t* opkb = sm + L::OP_KB + b * L::OP_KB_STRIDE;
        const uint32_t a_base = smem_u32(opa), kb_base = smem_u32(opkb);
        const uint32_t ap_base = smem_u32(sm + L::OP_A + bp * L::OP_A_STRIDE);
        const uint32_t kbp_base = smem_u32(sm + L::OP_KB + bp * L::OP_KB_STRIDE);

        // ---- CH1(c-1): X[bp] += [-W; Qh] Sm ----
        if (Q && tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem + TM_X0 + 128 * bp, sdesc_sw128(ap_base + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                         sdesc_sw128(sm_base + s * 2048, 16384, 1024), id, 1u);
            mma_commit(&bars[BAR_C1]);
        }

        // ---- E(c): gates and gated operands, in place in OP_A[b]; Kb -> OP_KB[b] ----
        if (P) {
            if (tid == 0) fl_la = fl_qk = false;
            wait_bar(BAR_LA);
            wait_bar(BAR_QK);
            float g0[16], g1[16];
            gate_load(reinterpret_cast<const float*>(sm + L::LA), D, Lc, tid, g0, g1);
            gate_chunk(g0, g1, opa, opkb, Lc, red, beta_s, beta_next, egm, egc + b * 128, egcm + b * 128, tid);
            if (tid == 0 && c + 1 < nch) {  // log_alpha staging consumed: fetch the next chunk's
                issue_la(c + 1);
                fl_la = true;
            }
            // V of this chunk: wait for its TMA; clear rows past the sequence end
            if (tid == 0) fl_v = false;
            wait_bar(BAR_V);
            if (Lc < C) {
                const int nz = (C - Lc) * 16;  // 16-byte chunks to clear
                for (int e = tid; e < nz; e += NT) {
                    const int r = Lc + (e >> 4), ch = e & 15;
                    *reinterpret_cast<uint4*>(sm + L::OP_V + (ch >> 3) * 8192 + sw128_chunk(r, ch & 7)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (tid < C) {  // prefetch the next chunk's beta
                const int64_t tn = t_begin + static_cast<int64_t>(c + 1) * C + tid;
                beta_next = (c + 1 < nch && tn < t_end) ? p.beta[tn * H + h] : 0.f;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*abort_s) break;

        // ---- MMA1(c): D = [Kh; Qh] Kb^T (128 x 64) ----
        if (P && tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem + TM_D, sdesc_sw128(a_base + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                         sdesc_sw128(kb_base + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024), id, s > 0);
            mma_commit(&bars[BAR_P1]);
        }
        // ---- U(c-1) -> OP_U once CH1 is done; the freed OP_A[bp] takes chunk c+1's q, k ----
        if (Q) {
            wait_bar(BAR_C1);
            tc_fence_after();
        }
        if (tid == 0 && c + 1 < nch) {
            issue_qk(c + 1);
            fl_qk = true;
        }
        if (Q && qw < 2) {
            const int r = 32 * qw + lane;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float a[32];
                tmem_ld32(tq + TM_X0 + 128 * bp + 64 * hw + 32 * part, a);
                tmem_ld_wait();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    *reinterpret_cast<uint4*>(sm + L::OP_U + hw * 8192 + sw128_chunk(r, 4 * part + ch)) =
                        pack8(a + 8 * ch);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- CH2(c-1): D_S = Kb^T U;  X[bp] += [0; M] U ----
        if (Q && tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_s = idesc_bf16_f32(128, 128, true, true);
            constexpr uint32_t id_o = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + TM_S, sdesc_sw128(kbp_base + s * 2048, 8192, 1024),
                         sdesc_sw128(u_base + s * 2048, 8192, 1024), id_s, s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + TM_X0 + 128 * bp, sdesc_sw128(a3_base + 8192 + s * 32, 16, 1024),
                         sdesc_sw128(u_base + s * 2048, 8192, 1024), id_o, 1u);
            mma_commit(&bars[BAR_C2]);
        }

        if (P) {
            // ---- D readout: N = Diag(beta) strict_lower(A) -> fp32 smem; Qh Kb^T kept in registers ----
            wait_bar(BAR_P1);
            tc_fence_after();
            {
                float a[32];
                tmem_ld32(tq + TM_D + 32 * hw, a);
                tmem_ld_wait();
                if (qw < 2) {
                    const int r = 32 * qw + lane;
                    store_n_row(Nf, r, hw, beta_s[r], a);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) mq[j] = a[j];
                }
            }
            tc_fence_before();
            __syncthreads();
            // ---- T = (I + N)^-1;  Tb = T Diag(beta) -> rows 0..63 of OP_A3 ----
            lower_inverse_tc(rows64(Nf), rows64(Tf), Xs, tid);
            store_tb(sm + L::OP_A3, rows64(Tf), beta_s, tid);
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            // ---- MMA3(c): D = [Tb; 0] Kh -> [W; 0];  X[b] = [Tb; 0] V -> [U0; 0] ----
            if (tid == 0) {
                tc_fence_after();
                constexpr uint32_t id = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + TM_D, sdesc_sw128(a3_base + s * 32, 16, 1024),
                             sdesc_sw128(a_base + s * 2048, 16384, 1024), id, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + TM_X0 + 128 * b, sdesc_sw128(a3_base + s * 32, 16, 1024),
                             sdesc_sw128(v_base + s * 2048, 8192, 1024), id, s > 0);
                mma_commit(&bars[BAR_P3]);
            }
        }

        // ---- state update and output of chunk c-1 (overlaps MMA3(c)) ----
        if (Q) {
            wait_bar(BAR_C2);
            tc_fence_after();
            const float dc = egc[bp * 128 + rho], dcm = egcm[bp * 128 + rho];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float a[32];
                tmem_ld32(tq + TM_S + 64 * hw + 32 * part, a);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) S[32 * part + j] = fmaf(dc, S[32 * part + j], dcm * a[j]);
            }
            if (qw >= 2) {
                const int rr = 32 * (qw - 2) + lane;
                const int64_t t0p = t_begin + static_cast<int64_t>(c - 1) * C;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    float a[32];
                    tmem_ld32(tq + TM_X0 + 128 * bp + 64 * hw + 32 * part, a);
                    tmem_ld_wait();
                    if (rr < Lprev) {
                        OutT* dst = static_cast<OutT*>(p.o) + ((t0p + rr) * H + h) * static_cast<int64_t>(D) +
                                    64 * hw + 32 * part;
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) store_out8<OutT>(dst + 8 * ch, a + 8 * ch);
                    }
                }
            }
        }
        if (P) {
            // M(c) = lower(Qh Kb^T) -> OP_A3 rows 128..191 (CH2(c-1) has finished reading the old M)
            if (qw >= 2) {
                const int rr = 32 * (qw - 2) + lane;
                store_m_row(sm + L::OP_A3, 128 + rr, rr, hw, mq);
            }
            wait_bar(BAR_P3);
            tc_fence_after();
            if (tid == 0 && c + 1 < nch) {  // V operand consumed: fetch the next chunk's
                issue_v(c + 1);
                fl_v = true;
            }
            // -W -> rows 0..63 of OP_A[b] (Kh no longer needed)
            if (qw < 2) {
                const int r = 32 * qw + lane;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    float a[32];
                    tmem_ld32(tq + TM_D + 64 * hw + 32 * part, a);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) a[j] = -a[j];
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
                        *reinterpret_cast<uint4*>(opa + hw * 16384 + sw128_chunk(r, 4 * part + ch)) = pack8(a + 8 * ch);
                }
            }
            // Sm = Diag(exp(gm)) S (state at the start of chunk c) -> OP_SM
            {
                const float sc = egm[rho];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float m8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) m8[e] = sc * S[8 * ch + e];
                    *reinterpret_cast<uint4*>(sm + L::OP_SM + hw * 16384 + sw128_chunk(rho, ch)) = pack8(m8);
                }
            }
            Lprev = Lc;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    // ---- wind down: every issued MMA and TMA has landed before TMEM and smem go away ----
    const bool aborted = *abort_s != 0;
    if (tid == 0) {
        mma_commit(&bars[BAR_FIN]);
        (void)mbar_wait(&bars[BAR_FIN], 0, kDrainLimit);
        if (aborted) {  // copies issued after the last wait on their barrier
            if (fl_la) (void)mbar_wait(&bars[BAR_LA], ph[BAR_LA], kDrainLimit);
            if (fl_qk) (void)mbar_wait(&bars[BAR_QK], ph[BAR_QK], kDrainLimit);
            if (fl_v) (void)mbar_wait(&bars[BAR_V], ph[BAR_V], kDrainLimit);
        }
    }
    if (p.S_final && !aborted) {
#pragma unroll
        for (int j = 0; j < 64; j += 4)
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

template <typename OutT>
cudaError_t launch_prefill_t(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_la, const PrefillArgs& a, cudaStream_t stream) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(kda_prefill_fused_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(Smem::ALLOC));
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const long long units = static_cast<long long>(a.num_seqs) * a.H;
    if (units == 0) return cudaSuccess;
    kda_prefill_fused_kernel<OutT><<<static_cast<unsigned>(units), NT, Smem::ALLOC, stream>>>(tm_q, tm_k, tm_v, tm_la, a);
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

cudaError_t launch_prefill_fused(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_la, const PrefillArgs& a, bool out_f32, cudaStream_t stream) {
    if (out_f32) return launch_prefill_t<float>(tm_q, tm_k, tm_v, tm_la, a, stream);
    return launch_prefill_t<__nv_bfloat16>(tm_q, tm_k, tm_v, tm_la, a, stream);
}

}  // namespace kda
