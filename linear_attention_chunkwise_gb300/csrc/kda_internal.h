// kda_internal.h -- launchers shared between the C-ABI front end and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/kda.h"

namespace kda {

// Debug builds (-DKDA_DEBUG_BOUNDS): before it touches memory, every CTA checks the ranges it derives
// from cu_seqlens, the schedule, the chunk table and snapshot entries (sequence, head, chunk and token
// ranges, snapshot entries) against the sizes of the buffers they index.  A range outside its buffer
// sets KDA_DEV_BOUNDS in the status word and the CTA skips that work; nothing traps.  Release builds
// compile the checks away (the condition is not evaluated).
#ifdef KDA_DEBUG_BOUNDS
#define KDA_BOUNDS(cond, status) (::kda::bounds_check((cond), (status)))
#else
#define KDA_BOUNDS(cond, status) true
#endif
#ifdef __CUDACC__
__device__ __forceinline__ bool bounds_check(bool ok, int32_t* status) {
    if (!ok && status) atomicOr(status, KDA_DEV_BOUNDS);
    return ok;
}
#endif

constexpr int kChunk = 64;   // chunk length of the prefill
constexpr int kHeadDim = 128;  // dk = dv

// KDA_OK when the current device is sm_103 (the only architecture the kernels are built for),
// KDA_ERR_UNSUPPORTED for another one, KDA_ERR_CUDA when the runtime cannot say.
kda_status device_check();

// ---- decode ----
struct DecodeFusion {  // KDA_FUSE_* bits and their parameters (see kda_fusion)
    uint32_t flags = 0;
    float l2_eps = 0.f, rms_eps = 0.f;
    const float* rms_weight = nullptr;
    const void* out_gate = nullptr;
};
cudaError_t launch_decode(bool f32_io, const void* q, const void* k, const void* v, const float* log_alpha,
                          const float* beta, float* S, int32_t num_slots, const int32_t* state_indices,
                          int32_t N, int32_t H, void* o, int32_t* device_status, cudaStream_t stream,
                          const DecodeFusion& fusion = DecodeFusion());

cudaError_t launch_decode_multi(bool f32_io, const void* q, const void* k, const void* v, const float* log_alpha,
                                const float* beta, float* S, int32_t num_slots, const int32_t* state_indices,
                                int32_t N, int32_t T, int32_t H, void* o, float* S_steps, int32_t* device_status,
                                cudaStream_t stream, const DecodeFusion& fusion = DecodeFusion());

// ---- prefill ----
struct PrefillArgs {
    const float* log_alpha;  // two-pass path's pass 1 reads it directly (the single pass by TMA)
    const float* beta;
    const float* S0;
    const int32_t* cu_seqlens;
    const int32_t* order;      // schedule: longest sequences first (workspace), or NULL (one sequence)
    const int32_t* chunk_off;  // two-pass path: chunk offsets [N + 2] (workspace)
    uint8_t* blobs;            // two-pass path: per (chunk, head) operand images (workspace)
    void* o;
    float* S_final;
    int32_t* device_status;
    int64_t total_tokens;
    int32_t num_seqs;
    int32_t H;
    int64_t blob_units = 0;  // two-pass path: (chunk, head) images the workspace holds
    // Two-pass path run in pieces: chunks [piece_begin, piece_begin + piece_len)
    // of every sequence; piece_len = 0 means all chunks in one launch pair.
    int32_t piece_begin = 0;
    int32_t piece_len = 0;
    // state snapshots (two-pass path): sorted (sequence, position) entries
    const int32_t* snap_seq = nullptr;
    const int32_t* snap_pos = nullptr;
    int32_t num_snaps = 0;
    float* S_snap = nullptr;
    // fused prologue (KDA_FUSE_L2NORM_QK, KDA_FUSE_BETA_SIGMOID: pass 1 applies them; the output
    // gate runs after the scan, launch_out_gate)
    uint32_t fuse_flags = 0;
    float l2_eps = 0.f;
};

// Bytes per (chunk, head) of the two-pass path's operand images:
// [-W; Qh] 32 KB | Kb 16 KB | Tb 8 KB | M 8 KB | exp(gm), exp(gC), exp(gC-gm) 1.5 KB.
constexpr size_t kPrefillBlobBytes = 67072;

// Sequence schedule (longest first) + cu_seqlens validation.
cudaError_t launch_schedule(const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t* order,
                            int32_t* device_status, cudaStream_t stream);

// fp32 -> bf16 copy (for fp32 q/k/v inputs).
cudaError_t launch_to_bf16(const float* src, void* dst, size_t n, cudaStream_t stream);

// Single-pass chunkwise prefill (one CTA per (sequence, head)); needs only
// the schedule as scratch.  q/k/v/log_alpha are read through TMA maps.
cudaError_t launch_prefill_fused(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                 const CUtensorMap& tm_la, const PrefillArgs& a, bool out_f32, cudaStream_t stream);

// Two-pass chunkwise prefill: chunk table, then per-(chunk, head) prep into
// the workspace, then the per-(sequence, head, dv slice) scan.
cudaError_t launch_chunk_table(const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t* chunk_off,
                               int32_t* device_status, const int32_t* snap_seq, const int32_t* snap_pos,
                               int32_t num_snaps, cudaStream_t stream);
// tm_snap: a map over S_snap as [num_snaps x H x 128 rows][128] fp32 (3-D, middle extent 1; at most
// kSnapMapRows rows, the rest stored without it), boxes of 32 rows x 32 columns, 128B-swizzled; any
// valid map when there are no snapshots.
constexpr int64_t kSnapMapRows = (int64_t{1} << 31) - 64;
cudaError_t launch_prefill_split(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                 const CUtensorMap& tm_snap, const PrefillArgs& a, int64_t max_chunks, bool out_f32,
                                 cudaStream_t stream);
// The two passes separately, for the piecewise schedule.  Pass 1's grid is
// `units` x H CTAs: units = chunk slots of the whole batch (piece_len = 0) or
// num_seqs x piece_len (piece mode); with beside_previous it is launched as a
// programmatic dependent of the previous launch on `stream` (a scan piece,
// whose CTAs release it once all of them run).  Pass 2 has num_seqs x H x 2 CTAs.
cudaError_t launch_chunk_prep(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const PrefillArgs& a, int64_t units,
                              cudaStream_t stream, bool beside_previous);
// y = RMSNorm(o) * w * gate in place on o ([rows, 128], the input dtype), w NULL = ones.
cudaError_t launch_out_gate(bool f32_io, void* o, const void* gate, const float* w, float eps, int64_t rows,
                            cudaStream_t stream);
cudaError_t launch_chunk_scan(const CUtensorMap& tm_v, const CUtensorMap& tm_snap, const PrefillArgs& a, bool out_f32,
                              cudaStream_t stream);

// Reverse-mode gradient of the prefill (kda_backward.cu).  Gradients are fp32,
// [T, H, 128] for q/k/v/log_alpha, [T, H] for beta, [N, H, 128, 128] for S0.
struct BackwardArgs {
    const void* q = nullptr;
    const void* k = nullptr;
    const void* v = nullptr;
    const float* log_alpha = nullptr;
    const float* beta = nullptr;
    const float* S0 = nullptr;
    const int32_t* cu_seqlens = nullptr;
    const int32_t* order = nullptr;      // sequences, longest first (NULL: in index order, one sequence)
    const int32_t* chunk_off = nullptr;  // chunk table
    const float* ckpt = nullptr;         // state after every chunk: entry (chunk_off[n] + c) x H + h
    const void* dO = nullptr;
    const float* dS_final = nullptr;
    float* dq = nullptr;
    float* dk = nullptr;
    float* dv = nullptr;
    float* dla = nullptr;
    float* dbeta = nullptr;
    float* dS0 = nullptr;
    float* rec = nullptr;        // per-(chunk, head) records of the prep kernel (backward_record_bytes each)
    float* xbuf = nullptr;       // adjoint of the state after every chunk, indexed like ckpt
    int32_t* device_status = nullptr;
    int64_t total_tokens = 0;
    int64_t chunk_slots = 0;     // chunk entries of ckpt, xbuf and rec
    int32_t num_seqs = 0;
    int32_t H = 0;
};
size_t backward_record_bytes();
// Snapshot entries at every chunk end (and sentinels up to max_entries) from the chunk table.
cudaError_t launch_ckpt_entries(const int32_t* cu_seqlens, const int32_t* chunk_off, int32_t N, int32_t max_entries,
                                int32_t* snap_seq, int32_t* snap_pos, int32_t* device_status, cudaStream_t stream);
// Fused prologue of the backward (q, k L2 norms, sigmoid beta into copies; inv = 1/norm of q and k
// per (token, head)) and the chain rule through it afterwards, in place on dq, dk, dbeta.
cudaError_t launch_bwd_prologue(bool f32_io, const void* q, const void* k, const float* beta, void* qh, void* kh,
                                float* bh, float* inv, int64_t rows, uint32_t flags, float eps, cudaStream_t stream);
cudaError_t launch_bwd_epilogue(bool f32_io, const void* q, const void* k, const float* bh, const float* inv,
                                float* dq, float* dk, float* dbeta, int64_t rows, uint32_t flags,
                                cudaStream_t stream);
// Backward of the output gate y = RMSNorm(o) * w * g for one grad_y (dy): dout = dL/do in the input dtype,
// dg = dL/dg fp32 [rows, 128], dw = dL/dw fp32 [128] (NULL: not computed) summed in a fixed order
// through dw_part (outgate_partial_bytes() of workspace).  w NULL means ones.
size_t outgate_partial_bytes();
cudaError_t launch_bwd_outgate(bool f32_io, const void* o, const void* g, const void* dy, const float* w, float eps,
                               void* dout, float* dg, float* dw, float* dw_part, int64_t rows, cudaStream_t stream);
// prep, scan, value and key kernels; chunk_slots bounds the batch's chunk count.
cudaError_t launch_backward(const BackwardArgs& a, bool f32_io, int64_t chunk_slots, cudaStream_t stream);

}  // namespace kda
