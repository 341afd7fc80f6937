// kda_prefill_split.cu -- two-pass chunkwise KDA prefill (tcgen05 + TMEM + TMA).
//
// Same chunk algebra as kda_prefill_common.cuh (derived from the KDA equation
// of "Understanding Kimi Delta Attention" (pyshine), "The KDA Recurrence", and
// the chunkwise form of its "The Chunkwise DPLR Algorithm" section), split so
// that the work that does NOT depend on the state runs fully in parallel:
//
//   pass 0  chunk table: chunk offsets of every sequence (from cu_seqlens).
//   pass 1  chunk prep, one CTA per (chunk, head), three CTAs per SM: gates,
//           Kh/Qh/Kb, MMA [Kh;Qh] Kb^T, the triangular inverse, Tb, M and
//           MMA W = Tb Kh.  It writes the scan's operands to the workspace as
//           ready-to-copy images of the swizzled shared-memory tiles:
//             [-W; Qh] (32 KB) | Kb (16 KB) | Tb (8 KB) | M (8 KB) |
//             exp(gm), exp(gC), exp(gC-gm) (3 x 512 B)
//   pass 2  scan, one CTA per (sequence, head, 64-column slice of dv): the
//           sequential chain only.  Per chunk it bulk-copies the images (one
//           chunk ahead into a second operand set; grids larger than one wave
//           use a single set, two CTAs per SM), TMA-loads its slice of v, and runs
//             X  = [Tb; 0] V + [-W; Qh] Sm      (= [U; Qh Sm])
//             D_S = Kb^T U,  X += [0; M] U      (= [U; O])
//             S <- Diag(exp(gC)) S + Diag(exp(gC-gm)) D_S
//           with the fp32 state slice in registers.
// Every on-chip wait is bounded; on expiry KDA_DEV_TIMEOUT is set and the
// CTA winds down instead of hanging.
#include <cuda_bf16.h>

#include <climits>

#include "kda_prefill_common.cuh"

namespace kda {
namespace {

using namespace pf;

constexpr uint32_t kBlobA = 0;          // [-W; Qh]
constexpr uint32_t kBlobKb = 32768;     // Kb
constexpr uint32_t kBlobTb = 49152;     // Tb (rows 0..63 of [Tb; M])
constexpr uint32_t kBlobM = 57344;      // M
constexpr uint32_t kBlobEv = 65536;     // exp(gm) | exp(gC) | exp(gC - gm), f32 [3][128]
static_assert(kBlobEv + 1536 == kPrefillBlobBytes, "blob layout");

// ---- bulk copy shared -> global (non-tensor), 16-byte aligned, sizes multiple of 16 ----
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
// PC consecutive TMEM columns of this thread's lane (32x32b shape): 32 or 16.
template <int PC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* r) {
    static_assert(PC == 32 || PC == 16, "32 or 16 columns");
    if (PC == 32) tmem_ld32(taddr, r);
    else tmem_ld16(taddr, r);
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// =========================================================== pass 0 ======
// chunk_off[n] = number of 64-token chunks in sequences 0..n-1, chunk_off[N]
// = total; chunk_off[N+1] = 1 when cu_seqlens is well formed (0 = c_0 <= ...
// <= c_N = total_tokens), else 0 and every offset 0 (nothing is computed).
__global__ void __launch_bounds__(1024) kda_chunk_table_kernel(const int32_t* __restrict__ cu, int32_t N,
                                                               int64_t total, int32_t* chunk_off,
                                                               int32_t* device_status, const int32_t* snap_seq,
                                                               const int32_t* snap_pos, int32_t num_snaps) {
    __shared__ int s_bad;
    __shared__ long long s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_bad = (cu[0] != 0 || static_cast<int64_t>(cu[N]) != total) ? 1 : 0;
    __syncthreads();
    const int per = (N + 1023) / 1024;
    const int i0 = min(N, tid * per), i1 = min(N, i0 + per);
    long long local = 0;
    bool bad = false;
    for (int n = i0; n < i1; ++n) {
        const int64_t a = cu[n], b = cu[n + 1];
        if (a < 0 || b < a || b > total) bad = true;
        else local += (b - a + C - 1) / C;
    }
    if (bad) atomicOr(&s_bad, 1);
    // block-wide exclusive scan of `local`
    long long incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long w = s_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    long long run = incl - local + (warp > 0 ? s_warp[warp - 1] : 0);
    const bool ok = s_bad == 0;
    for (int n = i0; n < i1; ++n) {
        chunk_off[n] = ok ? static_cast<int32_t>(run) : 0;
        if (ok) run += (static_cast<int64_t>(cu[n + 1]) - cu[n] + C - 1) / C;
    }
    if (tid == 1023) {
        chunk_off[N] = ok ? static_cast<int32_t>(s_warp[31]) : 0;
        chunk_off[N + 1] = ok ? 1 : 0;
    }
    if (tid == 0 && !ok && device_status) atomicOr(device_status, KDA_DEV_BAD_CU_SEQLENS);
    // snapshot entries: sequence in range, 0 < pos <= length, pos a multiple of the chunk or the
    // length, sorted by (sequence, position) without repeats
    if (ok && device_status) {
        bool bad_snap = false;
        for (int i = tid; i < num_snaps; i += 1024) {
            const int sq = snap_seq[i], ps = snap_pos[i];
            if (sq < 0 || sq >= N) { bad_snap = true; continue; }
            const int64_t len = static_cast<int64_t>(cu[sq + 1]) - cu[sq];
            if (ps <= 0 || ps > len || (ps % C != 0 && ps != len)) bad_snap = true;
            if (i > 0 && (snap_seq[i - 1] > sq || (snap_seq[i - 1] == sq && snap_pos[i - 1] >= ps))) bad_snap = true;
        }
        if (bad_snap) atomicOr(device_status, KDA_DEV_BAD_SNAPSHOT);
    }
}

// =========================================================== pass 1 ======
// Three CTAs per SM (the kernel is latency-bound: its throughput grows with
// the CTAs resident).  To fit, log_alpha goes straight from global memory to
// registers, and the parts of the image that are final after the gate phase
// (Qh, Kb, the exp vectors) are stored right away, so that their shared
// memory holds the inverse's fp32 scratch: N in the Kb tile, T in the two Qh
// halves, the partial sums and the block products in the Tb rows.
struct PrepSmem {
    static constexpr uint32_t OP_A = 0;          // [2 blk][128 rows][128 B]: [k;q] -> [Kh;Qh] -> [-W;Qh]
    static constexpr uint32_t T_LO = OP_A + 8192;           // f32 rows 0..31 of T (blk 0's Qh rows)
    static constexpr uint32_t T_HI = OP_A + 16384 + 8192;   // f32 rows 32..63 of T (blk 1's Qh rows)
    static constexpr uint32_t OP_KB = 32768;     // [2 blk][64 rows][128 B]: Kb, then f32 [64][64] N
    static constexpr uint32_t OP_A3 = 49152;     // [Tb (64 rows) | M (64 rows)] x 128 B
    static constexpr uint32_t XS = OP_A3;        // f32 inverse scratch (Tb rows, before Tb)
    static constexpr uint32_t RED = OP_A3 + 4096;  // f32 [8][128] gate partial sums (Tb rows, gate phase)
    static constexpr uint32_t EV = 65536;        // f32 [3][128]: exp(gm), exp(gC), exp(gC - gm)
    static constexpr uint32_t BETA = EV + 1536;  // f32 [64]
    static constexpr uint32_t BARS = BETA + 256;  // 2 x u64: q/k loaded, mma
    static constexpr uint32_t TMEM_SLOT = BARS + 16;
    static constexpr uint32_t TOTAL = TMEM_SLOT + 8;
    static constexpr uint32_t ALLOC = TOTAL + 1024;
};
static_assert(PrepSmem::XS + kInvScratchFloats * 4 <= PrepSmem::OP_A3 + 8192 &&
                  PrepSmem::RED + 4096 <= PrepSmem::OP_A3 + 8192,
              "scratch inside the Tb rows (the gate sums are dead before the inverse)");
static_assert(3 * (PrepSmem::ALLOC + 1024) <= 233472, "three prep CTAs must fit on one SM");

__global__ void __launch_bounds__(NT, 3)
    kda_chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const PrefillArgs p) {
    using L = PrepSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qw = warp & 3, hw = warp >> 2;
    const int H = p.H, N = p.num_seqs;
    const int32_t* co = p.chunk_off;
    const int unit = blockIdx.x / H;
    const int h = blockIdx.x - unit * H;
    if (co[N + 1] == 0) return;
    int j, seq;  // global chunk index, owning sequence
    if (p.piece_len > 0) {  // unit = (sequence, chunk of the piece)
        seq = unit / p.piece_len;
        const int c = p.piece_begin + (unit - seq * p.piece_len);
        if (seq >= N || c >= co[seq + 1] - co[seq]) return;
        j = co[seq] + c;
    } else {  // unit = global chunk; its sequence is the largest n with co[n] <= j
        j = unit;
        if (j >= co[N]) return;
        int lo = 0, hi = N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (co[mid] <= j) lo = mid;
            else hi = mid - 1;
        }
        seq = lo;
    }
    const int64_t t0 = static_cast<int64_t>(p.cu_seqlens[seq]) + static_cast<int64_t>(j - co[seq]) * C;
    const int64_t rem = p.cu_seqlens[seq + 1] - t0;
    const int Lc = static_cast<int>(rem < C ? rem : C);
    uint8_t* const blob = p.blobs + (static_cast<size_t>(j) * H + h) * kPrefillBlobBytes;
    if (!KDA_BOUNDS(seq >= 0 && seq < N && h < H && j >= 0 && (static_cast<int64_t>(j) + 1) * H <= p.blob_units &&
                        t0 >= 0 && Lc >= 1 && t0 + Lc <= p.total_tokens,
                    p.device_status))
        return;

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);  // 0: q/k, 1: mma
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::TMEM_SLOT);
    float* ev = reinterpret_cast<float*>(sm + L::EV);
    float* beta_s = reinterpret_cast<float*>(sm + L::BETA);
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bars[0], 4 * 8192);
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
            tma_load_3d(sm + L::OP_A + kh * 16384, &tm_k, &bars[0], 64 * kh, h, static_cast<int32_t>(t0));
            tma_load_3d(sm + L::OP_A + kh * 16384 + 8192, &tm_q, &bars[0], 64 * kh, h, static_cast<int32_t>(t0));
        }
    }
    // log_alpha rows of this thread, in flight while q and k land
    float4 g[8];
    gate_load4(p.log_alpha + (t0 * H + h) * D, H * D, Lc, tid, g);
    float beta_cur = (tid < Lc) ? p.beta[(t0 + tid) * H + h] : 0.f;
    if ((p.fuse_flags & KDA_FUSE_BETA_SIGMOID) && tid < Lc) beta_cur = 1.f / (1.f + expf(-beta_cur));
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    // Only thread 0 waits on each mbarrier; the others sleep in the block barrier that follows
    // (a spinning wait would take issue slots from the other CTAs on the SM).
    bool ok = true;
    if (tid == 0) ok = mbar_wait_pipe(&bars[0], 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tq = tmem + tmem_lane(qw);

    gate_chunk4(g, sm + L::OP_A, sm + L::OP_KB, Lc, reinterpret_cast<float*>(sm + L::RED), beta_s, beta_cur, ev,
                ev + 128, ev + 256, tid, (p.fuse_flags & KDA_FUSE_L2NORM_QK) != 0, p.l2_eps);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    const uint32_t a_base = smem_u32(sm + L::OP_A), kb_base = smem_u32(sm + L::OP_KB);
    const uint32_t a3_base = smem_u32(sm + L::OP_A3);
    if (tid == 0) {
        tc_fence_after();
        // D = [Kh; Qh] Kb^T  (128 x 64)
        constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
        for (int s = 0; s < 8; ++s)
            mma_bf16(tmem, sdesc_sw128(a_base + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                     sdesc_sw128(kb_base + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024), id, s > 0);
        mma_commit(&bars[1]);
        // the parts of the image that are final now: Qh (rows 64..127 of both blocks), Kb, exp vectors
        bulk_s2g(blob + kBlobA + 8192, sm + L::OP_A + 8192, 8192);
        bulk_s2g(blob + kBlobA + 16384 + 8192, sm + L::OP_A + 16384 + 8192, 8192);
        bulk_s2g(blob + kBlobKb, sm + L::OP_KB, 16384);
        bulk_s2g(blob + kBlobEv, sm + L::EV, 1536);
        bulk_commit();
    }
    if (tid == 0) {
        ok = mbar_wait_pipe(&bars[1], 0) && ok;
        bulk_wait_read();  // Qh and Kb have been read: their space becomes scratch
    }
    __syncthreads();
    tc_fence_after();
    float* Nf = reinterpret_cast<float*>(sm + L::OP_KB);
    const Rows64 Tf{reinterpret_cast<float*>(sm + L::T_LO), reinterpret_cast<float*>(sm + L::T_HI)};
    {
        float a[32];
        tmem_ld32(tq + 32 * hw, a);
        tmem_ld_wait();
        if (qw < 2) {
            const int r = 32 * qw + lane;
            store_n_row(Nf, r, hw, beta_s[r], a);
        } else {
            const int rr = 32 * (qw - 2) + lane;
            store_m_row(sm + L::OP_A3, 64 + rr, rr, hw, a);
        }
    }
    // The 16 x 16 diagonal blocks of T lie in the N rows a warp has just written: warp 0 holds rows and
    // columns 0..31 (blocks 0, 1), warp 5 rows and columns 32..63 (blocks 2, 3); each solves its two
    // blocks, a column per lane, without waiting for the other warps.
    if (warp == 0 || warp == 5) {
        __syncwarp();
        lower_inverse_diag_col(rows64(Nf), Tf, (warp == 0 ? 0 : 2) + (lane >> 4), lane & 15);
    }
    __syncthreads();
    lower_inverse_tc(rows64(Nf), Tf, reinterpret_cast<float*>(sm + L::XS), tid, true);
    store_tb(sm + L::OP_A3, Tf, beta_s, tid);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // [W; M Kh] = [Tb; M] Kh
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
        for (int s = 0; s < 4; ++s)
            mma_bf16(tmem, sdesc_sw128(a3_base + s * 32, 16, 1024), sdesc_sw128(a_base + s * 2048, 16384, 1024), id,
                     s > 0);
        mma_commit(&bars[1]);
    }
    if (tid == 0) ok = mbar_wait_pipe(&bars[1], 1) && ok;
    __syncthreads();
    tc_fence_after();
    if (qw < 2) {  // -W -> rows 0..63 of OP_A
        const int r = 32 * qw + lane;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float a[32];
            tmem_ld32(tq + 64 * hw + 32 * part, a);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = -a[e];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                *reinterpret_cast<uint4*>(sm + L::OP_A + hw * 16384 + sw128_chunk(r, 4 * part + ch)) = pack8(a + 8 * ch);
        }
    }
    if (!ok && tid == 0 && p.device_status) atomicOr(p.device_status, KDA_DEV_TIMEOUT);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(blob + kBlobA, sm + L::OP_A, 8192);                   // -W, block 0
        bulk_s2g(blob + kBlobA + 16384, sm + L::OP_A + 16384, 8192);   // -W, block 1
        bulk_s2g(blob + kBlobTb, sm + L::OP_A3, 16384);  // Tb and M, adjacent in both layouts
        bulk_commit();
        bulk_wait_read();  // shared memory may go once the copies have read it
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// =========================================================== pass 2 ======
constexpr int NV = 64;  // dv columns per scan CTA

// NSET operand sets: two (chunk c + 1's copies land while chunk c runs; one CTA per SM) or one
// (the copies follow the chunk's last use of the set; two CTAs per SM, each hiding the other's waits)
template <int NSET>
struct ScanSmemT {
    static constexpr uint32_t SET = 83968;       // 82 KB
    static constexpr uint32_t S_A = 0;           // [2 blk][128 rows][128 B]: [-W; Qh]
    static constexpr uint32_t S_KB = 32768;      // [2 blk][64 rows][128 B]: Kb
    static constexpr uint32_t S_A3 = 49152;      // [Tb | zeros | M] x 64 rows x 128 B
    static constexpr uint32_t S_V = 73728;       // [64 rows][128 B]: v slice (TMA, swizzled)
    static constexpr uint32_t S_EV = 81920;      // f32 [3][128]
    static constexpr uint32_t OP_SM = NSET * SET;  // [128 rows][128 B]: Sm slice
    static constexpr uint32_t OP_U = OP_SM + 16384;  // [64 rows][128 B]: U slice
    static constexpr uint32_t BARS = OP_U + 8192;    // 6 x u64: load0, load1, c1, c2, fin, c3
    static constexpr uint32_t TMEM_SLOT = BARS + 48;
    static constexpr uint32_t ABORT = TMEM_SLOT + 4;
    static constexpr uint32_t EVBAR = ABORT + 4;     // 2 x u64: a set's exp vectors landed (by chunk parity)
    static constexpr uint32_t TOTAL = EVBAR + 16;
    static constexpr uint32_t ALLOC = TOTAL + 1024;
};
using ScanSmem = ScanSmemT<2>;
static_assert(ScanSmem::EVBAR % 8 == 0 && ScanSmem::BARS % 8 == 0, "mbarriers are 8-byte aligned");
// two one-set CTAs (and the 1 KB the runtime reserves for each) in the SM's 228 KB
static_assert(2 * (ScanSmemT<1>::ALLOC + 1024) <= 233472, "two one-set scan CTAs per SM");
// per-warp staging inside a consumed operand set: the state slice (128 rows x 64 fp32 over all warps)
// fits the [-W; Qh] tile, the output rows (64 rows x 64 columns, at most fp32) the Kb tile
static_assert(128 * 64 * 4 <= ScanSmem::S_KB - ScanSmem::S_A, "state stage over the [-W; Qh] tile");
static_assert(64 * 64 * 4 <= ScanSmem::S_A3 - ScanSmem::S_KB, "output stage over the Kb tile");
static_assert(ScanSmem::ALLOC <= 232448, "scan shared memory over the per-CTA limit");
constexpr uint32_t kLoadBytes = 32768 + 16384 + 8192 + 8192 + 1536 + 8192;

// Store a warp's 32 x PC block of the state (lane = block row, PC consecutive columns) to global
// memory, `dst` = the block's first row, rows D floats apart.  The block is transposed through the
// warp's own 32 x PC floats of shared memory (16-byte chunks xor-swizzled by the row), so each store
// instruction writes whole PC * 4-byte row segments of 32 / (PC / 4) rows instead of 16 bytes in each
// of 32 rows.
// The staging alone: lane = block row, row r's 16-byte chunk j at position j ^ (r mod CH).  For PC = 32
// (128-byte rows) on a 1024-byte aligned stage this is the 128B-swizzled layout of a tensor copy's box.
template <int PC>
__device__ __forceinline__ void stage_state_rows(const float (&S)[PC], float* stage, int lane) {
    constexpr int CH = PC / 4;
#pragma unroll
    for (int j = 0; j < CH; ++j)
        *reinterpret_cast<float4*>(stage + lane * PC + 4 * (j ^ (lane & (CH - 1)))) =
            make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
}
template <int PC>
__device__ __forceinline__ void store_state_rows(float* dst, const float (&S)[PC], float* stage, int lane) {
    constexpr int CH = PC / 4;    // 16-byte chunks per row
    constexpr int RPI = 32 / CH;  // rows per store instruction
    stage_state_rows<PC>(S, stage, lane);
    __syncwarp();
    const int rr = lane / CH, j = lane % CH;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int r = i * RPI + rr;
        *reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * D + 4 * j) =
            *reinterpret_cast<const float4*>(stage + r * PC + 4 * (j ^ (r & (CH - 1))));
    }
    __syncwarp();
}

// The reverse of store_state_rows: whole row segments from global memory, transposed through the
// warp's shared memory into lane = block row, PC consecutive columns.
template <int PC>
__device__ __forceinline__ void load_state_rows(const float* src, float (&S)[PC], float* stage, int lane) {
    constexpr int CH = PC / 4;
    constexpr int RPI = 32 / CH;
    const int rr = lane / CH, j = lane % CH;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int r = i * RPI + rr;
        *reinterpret_cast<float4*>(stage + r * PC + 4 * (j ^ (r & (CH - 1)))) =
            *reinterpret_cast<const float4*>(src + static_cast<size_t>(r) * D + 4 * j);
    }
    __syncwarp();
#pragma unroll
    for (int jj = 0; jj < CH; ++jj) {
        const float4 t = *reinterpret_cast<const float4*>(stage + lane * PC + 4 * (jj ^ (lane & (CH - 1))));
        S[4 * jj] = t.x; S[4 * jj + 1] = t.y; S[4 * jj + 2] = t.z; S[4 * jj + 3] = t.w;
    }
    __syncwarp();
}

// Store a warp's 32 output rows (lane = row, PC consecutive columns as fp32) to `dst` (row 0, rows
// `row_stride` elements apart; only rows < nrows), converted to OutT, as whole row segments: the
// packed rows are transposed through the warp's PC * sizeof(OutT) * 32 bytes of shared memory
// (16-byte chunks xor-swizzled so both passes are conflict-free).
template <typename OutT, int PC>
__device__ __forceinline__ void store_out_rows(OutT* dst, int64_t row_stride, int nrows, const float (&a)[PC],
                                               uint8_t* stage, int lane) {
    constexpr int RB = PC * static_cast<int>(sizeof(OutT));  // bytes per row
    constexpr int CH = RB / 16;                               // 16-byte chunks per row
    constexpr int RPI = 32 / CH;                              // rows per store instruction
    constexpr int SH = RB >= 128 ? 0 : (RB == 64 ? 1 : 2);    // rows sharing one 128-byte bank line
    static_assert(CH >= 2 && CH <= 8, "row segment of 32 to 128 bytes");
    const int key = (lane >> SH) & (CH - 1);
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
        uint4 pk;
        if constexpr (sizeof(OutT) == 2) {
            pk = pack8(a + 8 * ch);
        } else {
            pk = make_uint4(__float_as_uint(a[4 * ch]), __float_as_uint(a[4 * ch + 1]), __float_as_uint(a[4 * ch + 2]),
                            __float_as_uint(a[4 * ch + 3]));
        }
        *reinterpret_cast<uint4*>(stage + lane * RB + 16 * (ch ^ key)) = pk;
    }
    __syncwarp();
    const int rr = lane / CH, j = lane % CH;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int r = i * RPI + rr;
        if (r < nrows)
            *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(dst + r * row_stride) + 16 * j) =
                *reinterpret_cast<const uint4*>(stage + r * RB + 16 * (j ^ ((r >> SH) & (CH - 1))));
    }
    __syncwarp();
}

// NTS threads in NTS/128 column groups (256: two groups of 32 state columns per thread; 512: four
// of 16).  Thread (warp w): lane quarter qw = w % 4 (state rows 32 qw + lane, the TMEM lanes it may
// read), column group cq = w / 4.
template <typename OutT, int NTS, int NSET>
__global__ void __launch_bounds__(NTS, 3 - NSET)
    kda_chunk_scan_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_snap,
                          const PrefillArgs p) {
    using L = ScanSmemT<NSET>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int CQ = NTS / 128;  // column groups
    constexpr int PC = NV / CQ;    // state columns per thread
    const int qw = warp & 3, cq = warp >> 2;
    const int H = p.H, N = p.num_seqs;
    const int32_t* co = p.chunk_off;
    constexpr int NSLICE = D / NV;
    const int slice = blockIdx.x % NSLICE;
    const int h = (blockIdx.x / NSLICE) % H;
    const int pos = blockIdx.x / (NSLICE * H);
    // A pass-1 launch queued behind this one as its programmatic dependent may start once every CTA of
    // this grid has reached here: it then only takes the SMs the scan leaves idle.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (co[N + 1] == 0) return;  // malformed cu_seqlens: nothing is written
    const int seq = p.order ? p.order[pos] : pos;
    const int nch_seq = co[seq + 1] - co[seq];
    // chunks [cb, cb + nch) of the sequence; in piece mode the state enters
    // from S_final (the previous piece's carry) unless the piece is the first
    int cb = 0, nch = nch_seq;
    if (p.piece_len > 0) {
        cb = p.piece_begin;
        if (cb > 0 && cb >= nch_seq) return;
        nch = min(nch_seq - cb, p.piece_len);
        if (nch < 0) nch = 0;
    }
    const int64_t t_begin = p.cu_seqlens[seq] + static_cast<int64_t>(cb) * C, t_end = p.cu_seqlens[seq + 1];
    const int jb = co[seq] + cb;
    const int j0 = slice * NV;
    const float* S_in = cb == 0 ? p.S0 : p.S_final;
    // snapshot entries of this sequence (sorted by sequence, then position): [si, se)
    int si = 0, se = 0;
    if (p.num_snaps > 0) {
        int lo = 0, hi = p.num_snaps;  // first entry with sequence >= seq
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (p.snap_seq[mid] < seq) lo = mid + 1;
            else hi = mid;
        }
        si = lo;
        hi = p.num_snaps;  // first entry with sequence > seq
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (p.snap_seq[mid] <= seq) lo = mid + 1;
            else hi = mid;
        }
        se = lo;
        while (si < se && p.snap_pos[si] <= cb * C) ++si;  // taken by an earlier piece
    }
    const int64_t seq_len = static_cast<int64_t>(p.cu_seqlens[seq + 1]) - p.cu_seqlens[seq];
    int next_snap = si < se ? p.snap_pos[si] : INT_MAX;
    if (!KDA_BOUNDS(seq >= 0 && seq < N && h < H && t_begin >= 0 && t_end <= p.total_tokens && seq_len >= 0 &&
                        static_cast<int64_t>(nch_seq) * C >= seq_len && static_cast<int64_t>(nch_seq) * C < seq_len + C &&
                        cb >= 0 && nch >= 0 && cb + nch <= nch_seq && jb >= 0 &&
                        (static_cast<int64_t>(jb) + nch) * H <= p.blob_units && 0 <= si && si <= se &&
                        se <= p.num_snaps,
                    p.device_status))
        return;

    // state: row rho, columns [j0 + PC*cq, +PC)
    const int rho = 32 * qw + lane;
    float S[PC];
    const size_t srow = ((static_cast<size_t>(seq) * H + h) * D + rho) * D + j0 + PC * cq;
    if (S_in) {  // staged in operand set 0, which the first copies fill only after the block barrier below
        load_state_rows<PC>(S_in + ((static_cast<size_t>(seq) * H + h) * D + 32 * qw) * D + j0 + PC * cq, S,
                            reinterpret_cast<float*>(sm) + warp * 32 * PC, lane);
    } else {
#pragma unroll
        for (int j = 0; j < PC; ++j) S[j] = 0.f;
    }
    if (nch == 0) {
        if (p.S_final) {
#pragma unroll
            for (int j = 0; j < PC; j += 4)
                *reinterpret_cast<float4*>(p.S_final + srow + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
        return;
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* evbar = reinterpret_cast<uint64_t*>(sm + L::EVBAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::TMEM_SLOT);
    volatile int* abort_s = reinterpret_cast<volatile int*>(sm + L::ABORT);
    if (tid == 0) {
        *abort_s = 0;
        for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
        mbar_init(&evbar[0], 1);
        mbar_init(&evbar[1], 1);
        fence_mbar_init();
        prefetch_tmap(&tm_v);
        if (p.num_snaps > 0) prefetch_tmap(&tm_snap);
    }
    for (int e = tid; e < NSET * 512; e += NTS)  // zero rows of every set's [Tb | 0 | M] tile
        reinterpret_cast<uint4*>(sm + (e >> 9) * L::SET + L::S_A3 + 8192)[e & 511] = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tq = tmem + tmem_lane(qw);
    constexpr uint32_t TM_X = 0;    // + 64 * parity
    constexpr uint32_t TM_DS = 128;

    auto issue_loads = [&](int c) {
        const int sb = c % NSET;
        uint8_t* set = sm + sb * L::SET;
        uint64_t* bar = &bars[sb];
        const uint8_t* blob = p.blobs + (static_cast<size_t>(jb + c) * H + h) * kPrefillBlobBytes;
        // the exp vectors first, on their own barrier: the state conversion needs only them
        mbar_arrive_expect_tx(&evbar[sb], 1536);
        bulk_g2s(set + L::S_EV, blob + kBlobEv, 1536, &evbar[sb]);
        mbar_arrive_expect_tx(bar, kLoadBytes - 1536);
        bulk_g2s(set + L::S_A, blob + kBlobA, 32768, bar);
        bulk_g2s(set + L::S_KB, blob + kBlobKb, 16384, bar);
        bulk_g2s(set + L::S_A3, blob + kBlobTb, 8192, bar);
        bulk_g2s(set + L::S_A3 + 16384, blob + kBlobM, 8192, bar);
        tma_load_3d(set + L::S_V, &tm_v, bar, j0, h, static_cast<int32_t>(t_begin + static_cast<int64_t>(c) * C));
    };
    if (tid == 0) {
        issue_loads(0);
        if (NSET == 2 && nch > 1) issue_loads(1);
    }
    uint32_t ph_load = 0, ph_c1 = 0, ph_c2 = 0, ph_c3 = 0;  // ph_load: parity of bars[i] (and evbar[i]) in bit i
    auto wait_bar = [&](uint64_t* bar, uint32_t& ph) {
        if (!mbar_wait_pipe(bar, ph)) *abort_s = 1;
        ph ^= 1u;
    };
    const uint64_t d_sm = sdesc_sw128(smem_u32(sm + L::OP_SM), 8192, 1024);
    const uint64_t d_u = sdesc_sw128(smem_u32(sm + L::OP_U), 8192, 1024);

    int c_stop = nch;  // the step the loop stopped at (nch when it ran to the end)
    for (int c = 0; c < nch; ++c) {
        const int b = c & 1;               // TMEM half of this chunk's X
        const int sb = NSET == 2 ? b : 0;  // its operand set
        uint8_t* set = sm + sb * L::SET;
        const float* evs = reinterpret_cast<const float*>(set + L::S_EV);
        const int64_t t0 = t_begin + static_cast<int64_t>(c) * C;
        const int Lc = static_cast<int>(t_end - t0 < C ? t_end - t0 : C);
        // Every thread waits for the exp vectors only; the state conversion below overlaps the rest
        // of the copies, which thread 0 waits for before the block barrier (all threads in the last,
        // ragged chunk, whose v rows past the sequence end they clear).
        const uint32_t par = (ph_load >> sb) & 1u;
        ph_load ^= 1u << sb;
        if (Lc < C) {  // rows of v past the sequence end -> 0
            if (!mbar_wait_pipe(&bars[sb], par)) *abort_s = 1;
            for (int e = tid; e < (C - Lc) * 8; e += NTS) {
                const int r = Lc + (e >> 3);
                *reinterpret_cast<uint4*>(set + L::S_V + sw128_chunk(r, e & 7)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (!mbar_wait_pipe(&evbar[sb], par)) *abort_s = 1;
        {  // Sm = Diag(exp(gm)) S -> OP_SM (row rho, chunks PC*cq/8 ..)
            const float sc = evs[rho];
#pragma unroll
            for (int ch = 0; ch < PC / 8; ++ch) {
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = sc * S[8 * ch + e];
                *reinterpret_cast<uint4*>(sm + L::OP_SM + sw128_chunk(rho, PC * cq / 8 + ch)) = pack8(m8);
            }
        }
        fence_async_smem();
        if (Lc == C && tid == 0 && !mbar_wait_pipe(&bars[sb], par)) *abort_s = 1;
        tc_fence_before();
        __syncthreads();
        if (*abort_s) {  // a bounded wait expired: every thread sees it after the barrier
            c_stop = c;
            break;
        }
        // shared-memory descriptors; a K-step adds its byte offset / 16 to the start-address field
        const uint64_t d_a = sdesc_sw128(smem_u32(set + L::S_A), 16, 1024);
        const uint64_t d_kb = sdesc_sw128(smem_u32(set + L::S_KB), 8192, 1024);
        const uint64_t d_a3 = sdesc_sw128(smem_u32(set + L::S_A3), 16, 1024);
        const uint64_t d_v = sdesc_sw128(smem_u32(set + L::S_V), 8192, 1024);
        const uint32_t tx = tmem + TM_X + 64 * b;
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, NV, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)  // X = [Tb; 0] V
                mma_bf16(tx, d_a3 + 2 * s, d_v + 128 * s, id, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)  // X += [-W; Qh] Sm
                mma_bf16(tx, d_a + (s >> 2) * 1024 + (s & 3) * 2, d_sm + 128 * s, id, 1u);
            mma_commit(&bars[2]);
        }
        // the other set held chunk c-1, consumed by the end of the previous step: fetch chunk c+1
        // (a warp other than the MMA issuer issues the copies)
        if (NSET == 2 && tid == 32 && c >= 1 && c + 1 < nch) issue_loads(c + 1);
        wait_bar(&bars[2], ph_c1);
        tc_fence_after();
        if (qw < 2) {  // U -> OP_U (row r, chunks PC*cq/8 ..)
            const int r = 32 * qw + lane;
            float a[PC];
            tmem_ld_cols<PC>(tq + TM_X + 64 * b + PC * cq, a);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < PC / 8; ++ch)
                *reinterpret_cast<uint4*>(sm + L::OP_U + sw128_chunk(r, PC * cq / 8 + ch)) = pack8(a + 8 * ch);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_s = idesc_bf16_f32(128, NV, true, true);
            constexpr uint32_t id_o = idesc_bf16_f32(128, NV, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)  // D_S = Kb^T U
                mma_bf16(tmem + TM_DS, d_kb + 128 * s, d_u + 128 * s, id_s, s > 0);
            mma_commit(&bars[3]);  // the state update needs only D_S
#pragma unroll
            for (int s = 0; s < 4; ++s)  // X += [0; M] U  (zero rows, then M, at 8 KB into the tile)
                mma_bf16(tx, d_a3 + 512 + 2 * s, d_u + 128 * s, id_o, 1u);
            mma_commit(&bars[5]);  // the output rows
        }
        wait_bar(&bars[3], ph_c2);
        tc_fence_after();
        {
            const float dc = evs[128 + rho], dcm = evs[256 + rho];
            float a[PC];
            tmem_ld_cols<PC>(tq + TM_DS + PC * cq, a);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < PC; ++e) S[e] = fmaf(dc, S[e], dcm * a[e]);
        }
        bool snap_stored = false;
        {  // state snapshots at the end of this chunk (positions are sequence-relative): each warp stages its
           // 32 x 32 block in this chunk's operand set (its MMAs have completed) in the 128B-swizzled
           // layout of the snapshot map's box, and its lane 0 stores it with one tensor copy
            const int64_t done = min(static_cast<int64_t>(cb + c + 1) * C, seq_len);
            while (next_snap <= done) {
                if (next_snap == done) {
                    float* stage = reinterpret_cast<float*>(set) + warp * 32 * PC;
                    const int64_t row = (static_cast<int64_t>(si) * H + h) * D + 32 * qw;
                    if (snap_stored && lane == 0) bulk_wait_read();  // a second entry at the same position
                    __syncwarp();
                    if (row + 32 <= kSnapMapRows) {  // the map's coordinates are 32-bit
                        stage_state_rows<PC>(S, stage, lane);
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tm_snap, stage, j0 + PC * cq, 0, static_cast<int32_t>(row));
                            bulk_commit();
                        }
                        snap_stored = true;
                    } else {
                        store_state_rows<PC>(p.S_snap + row * D + j0 + PC * cq, S, stage, lane);
                    }
                }
                ++si;
                next_snap = si < se ? p.snap_pos[si] : INT_MAX;
            }
        }
        if (qw >= 2) {  // O rows -> global
            wait_bar(&bars[5], ph_c3);
            tc_fence_after();
            float a[PC];
            tmem_ld_cols<PC>(tq + TM_X + 64 * b + PC * cq, a);
            tmem_ld_wait();
            // staged in this chunk's Kb tile (its MMAs have completed; every load of the set
            // rewrites it), beside the [-W; Qh] tile the state snapshot may use -- never in the
            // zero rows of [Tb | 0 | M], which are written once
            const int row0 = 32 * (qw - 2);
            store_out_rows<OutT, PC>(
                static_cast<OutT*>(p.o) + ((t0 + row0) * H + h) * static_cast<int64_t>(D) + j0 + PC * cq,
                static_cast<int64_t>(H) * D, Lc - row0, a, set + L::S_KB + ((qw - 2) + 2 * cq) * (32 * PC * 4),
                lane);
        }
        if (snap_stored && lane == 0) bulk_wait_read();  // the snapshot copies have read the staged blocks
        if (NSET == 1 && c + 1 < nch) {  // every read of the set (MMAs, staging) is done: refill it
            fence_async_smem();
            __syncthreads();
            if (tid == 32) issue_loads(c + 1);
        }
        tc_fence_before();
    }
    __syncthreads();
    const bool ok = *abort_s == 0;
    if (!ok && tid == 0 && p.device_status) atomicOr(p.device_status, KDA_DEV_TIMEOUT);
    if (tid == 0) {  // every MMA and copy this CTA issued has landed before it exits
        mma_commit(&bars[4]);
        (void)mbar_wait(&bars[4], 0, kDrainLimit);
        // a step's loads are waited for (to completion) in that step; the next chunk's are issued
        // after the step's barrier (one set: at its end), so only a stop at step 0 of the two-set form
        // leaves chunk 1's (issued up front) in flight
        if (NSET == 2 && c_stop == 0 && nch > 1) {
            (void)mbar_wait(&evbar[1], 0, kDrainLimit);
            (void)mbar_wait(&bars[1], 0, kDrainLimit);
        }
    }
    if (p.S_final && ok)  // staged in operand set 0: every copy into it has been consumed
        store_state_rows<PC>(p.S_final + ((static_cast<size_t>(seq) * H + h) * D + 32 * qw) * D + j0 + PC * cq, S,
                             reinterpret_cast<float*>(sm) + warp * 32 * PC, lane);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// Sets one function attribute on first use per device.
template <typename K>
cudaError_t set_attr_once(K kernel, cudaFuncAttribute attr, int value, int* configured) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64 && configured[dev]) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, attr, value);
    if (err == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = 1;
    return err;
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes, int* configured) {
    return set_attr_once(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes), configured);
}

}  // namespace

cudaError_t launch_chunk_table(const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t* chunk_off,
                               int32_t* device_status, const int32_t* snap_seq, const int32_t* snap_pos,
                               int32_t num_snaps, cudaStream_t stream) {
    kda_chunk_table_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, num_seqs, total_tokens, chunk_off, device_status,
                                                   snap_seq, snap_pos, num_snaps);
    return cudaGetLastError();
}

cudaError_t launch_chunk_prep(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const PrefillArgs& a, int64_t units,
                              cudaStream_t stream, bool beside_previous) {
    static int cfg_prep[64];
    cudaError_t err = set_smem(kda_chunk_prep_kernel, PrepSmem::ALLOC, cfg_prep);
    if (err != cudaSuccess) return err;
    static int carveout_prep[64];  // all of the unified L1 as shared memory: three CTAs per SM
    err = set_attr_once(kda_chunk_prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                        cudaSharedmemCarveoutMaxShared, carveout_prep);
    if (err != cudaSuccess) return err;
    const long long prep_ctas = static_cast<long long>(units) * a.H;
    if (prep_ctas > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(prep_ctas));
        cfg.blockDim = dim3(NT);
        cfg.dynamicSmemBytes = PrepSmem::ALLOC;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        if (beside_previous) {  // programmatic dependent of the previous launch (a scan piece): it reads
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // nothing that one writes
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        err = cudaLaunchKernelEx(&cfg, kda_chunk_prep_kernel, tm_q, tm_k, a);
    }
    return err;
}

cudaError_t launch_prefill_split(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                 const CUtensorMap& tm_snap, const PrefillArgs& a, int64_t max_chunks, bool out_f32,
                                 cudaStream_t stream) {
    const cudaError_t err = launch_chunk_prep(tm_q, tm_k, a, max_chunks, stream, false);
    if (err != cudaSuccess) return err;
    return launch_chunk_scan(tm_v, tm_snap, a, out_f32, stream);
}

template <typename OutT, int NSET>
cudaError_t launch_scan_t(const CUtensorMap& tm_v, const CUtensorMap& tm_snap, const PrefillArgs& a, unsigned ctas,
                          cudaStream_t stream) {
    constexpr int NTS = 256;  // 512 threads (16 columns each) measured no faster: the chunk is not epilogue-bound
    constexpr uint32_t alloc = ScanSmemT<NSET>::ALLOC;
    static int configured[64];
    cudaError_t err = set_smem(kda_chunk_scan_kernel<OutT, NTS, NSET>, alloc, configured);
    if (err != cudaSuccess) return err;
    if (NSET == 1) {  // all of the unified L1 as shared memory: two CTAs per SM
        static int carveout[64];
        err = set_attr_once(kda_chunk_scan_kernel<OutT, NTS, NSET>, cudaFuncAttributePreferredSharedMemoryCarveout,
                            cudaSharedmemCarveoutMaxShared, carveout);
        if (err != cudaSuccess) return err;
    }
    kda_chunk_scan_kernel<OutT, NTS, NSET><<<ctas, NTS, alloc, stream>>>(tm_v, tm_snap, a);
    return cudaGetLastError();
}

// One scan CTA per (sequence, head, dv slice).  A grid that fits the GPU at one CTA per SM runs the
// two-set form (each chain at its shortest).  A larger one runs the one-set form, two CTAs per SM,
// where that pays (A/B, 32 heads, bitwise-equal outputs): when the grid fits at two per SM (3 x 8192
// tokens: 0.821 against 0.842 ms, the two-set form leaving a tail wave of whole chains), or when the
// sequences average at most 32 chunks, so each CTA's start (state, first copies) is hidden behind the
// other's chain (64 x 1024 tokens: 1.87 against 2.00 ms).  Longer sequences in several waves keep
// the two-set form (16 x 4096 tokens: 1.82 against 1.87 ms; the varlen mix of 1k-64k tokens even).
cudaError_t launch_chunk_scan(const CUtensorMap& tm_v, const CUtensorMap& tm_snap, const PrefillArgs& a, bool out_f32,
                              cudaStream_t stream) {
    const long long scan_ctas = static_cast<long long>(a.num_seqs) * a.H * (D / NV);
    if (scan_ctas == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const unsigned n = static_cast<unsigned>(scan_ctas);
    const bool short_chains = a.total_tokens <= static_cast<int64_t>(32 * C) * a.num_seqs;
    if (scan_ctas > sms && (scan_ctas <= 2LL * sms || short_chains))
        return out_f32 ? launch_scan_t<float, 1>(tm_v, tm_snap, a, n, stream)
                       : launch_scan_t<__nv_bfloat16, 1>(tm_v, tm_snap, a, n, stream);
    return out_f32 ? launch_scan_t<float, 2>(tm_v, tm_snap, a, n, stream)
                   : launch_scan_t<__nv_bfloat16, 2>(tm_v, tm_snap, a, n, stream);
}

// ============================================================ output gate ==
// y = o / sqrt(mean_c o_c^2 + eps) * w * g, in place on o, after the scan: the output gate of "kimi
// delta attn from first principles" (aryagxr), "KDA has three gates".  One warp per (token, head)
// row, 4 channels per lane; the row's mean square is taken from the row itself, so the scan needs
// no cross-slice exchange.  Grid-stride over the rows (8k: 30.6 us at 65 % of DRAM peak; loading four
// rows per warp before reducing any measured slower, 8k with the gate 344 -> 360 us).
namespace {
__device__ __forceinline__ float4 og_ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 og_ld4(const __nv_bfloat16* p) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u), __uint_as_float(r.y << 16),
                       __uint_as_float(r.y & 0xffff0000u));
}
__device__ __forceinline__ void og_st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void og_st4(__nv_bfloat16* p, float4 v) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
}

template <typename IoT>
__global__ void __launch_bounds__(256) kda_out_gate_kernel(IoT* o, const IoT* __restrict__ g,
                                                           const float* __restrict__ w, float eps, int64_t rows) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 wv = w ? make_float4(w[4 * lane], w[4 * lane + 1], w[4 * lane + 2], w[4 * lane + 3])
                        : make_float4(1.f, 1.f, 1.f, 1.f);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp; row < rows;
         row += static_cast<int64_t>(gridDim.x) * 8) {
        const size_t off = static_cast<size_t>(row) * kHeadDim + 4 * lane;
        const float4 ov = og_ld4(o + off), gv = og_ld4(g + off);
        float ss = ov.x * ov.x + ov.y * ov.y + ov.z * ov.z + ov.w * ov.w;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
        const float r = rsqrtf(ss * (1.f / kHeadDim) + eps);
        og_st4(o + off, make_float4(ov.x * r * wv.x * gv.x, ov.y * r * wv.y * gv.y, ov.z * r * wv.z * gv.z,
                                    ov.w * r * wv.w * gv.w));
    }
}
}  // namespace

cudaError_t launch_out_gate(bool f32_io, void* o, const void* gate, const float* w, float eps, int64_t rows,
                            cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const int64_t need = (rows + 7) / 8;
    const unsigned blocks = static_cast<unsigned>(need < 8LL * sms ? need : 8LL * sms);
    if (f32_io)
        kda_out_gate_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<float*>(o), static_cast<const float*>(gate),
                                                               w, eps, rows);
    else
        kda_out_gate_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<__nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(gate), w, eps, rows);
    return cudaGetLastError();
}


}  // namespace kda
