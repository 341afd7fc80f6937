/*
 * kda.h -- C ABI of libkda: Kimi Delta Attention (KDA) recurrence on sm_103a.
 *
 * The operation (per head, state S is dk x dv, rows = key channels):
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t                         (read from the UPDATED state)
 *
 * Sources: the KDA equation in "Understanding Kimi Delta Attention"
 * (pyshine), section "The KDA Recurrence: Scalar Gate vs Channel-wise Gate";
 * per-row (key-channel) decay and the read o_t = S_t^T q_t in "kimi delta
 * attn from first principles" (aryagxr), section "KDA".  Page 1 of the
 * sources reads the state with k_t instead ("Understanding the
 * Recurrence"); this library follows the query read.
 *
 * Conventions shared by every entry point
 *   - alpha_t = exp(log_alpha_t) (natural log), one gate per key channel;
 *     beta_t is used as given (the sources give it as a sigmoid in [0, 1]).
 *   - No scaling or normalisation of q/k in the plain entry points: callers
 *     pass q and k already L2-normalised per (token, head), as the sources'
 *     "KDA Architecture" section describes (the _ex entry points can do it
 *     inside the kernels, see kda_fusion).
 *   - dk = dv = 128 only (the sources' 128 x 128 state); anything else
 *     returns KDA_ERR_UNSUPPORTED.
 *   - All tensors are dense, row-major, caller-owned DEVICE memory.  q, k,
 *     v, log_alpha, o and the states are 16-byte aligned; beta, cu_seqlens,
 *     state_indices and device_status 4-byte aligned; the prefill workspace
 *     256-byte aligned.  The library allocates no device memory, never
 *     synchronises the host, and enqueues all work on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream).  It owns no streams,
 *     events or locks and keeps no state between calls except, per device,
 *     the kernels' attribute settings, the entry points it looks up in the
 *     driver, and (kda_prefill_noalloc only) its fixed scratch array.
 *   - Argument errors are returned synchronously before anything is
 *     enqueued.  Data-dependent errors found on the device are OR-ed into
 *     *device_status (if non-NULL) as KDA_DEV_* bits; the affected sequences
 *     or slots are skipped and nothing is written out of bounds.  The caller
 *     reads *device_status after the stream completes and should zero it
 *     before the call.
 *   - Calls on different streams that write the same buffers race.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 1

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

typedef struct CUstream_st *kda_stream_t; /* same type as cudaStream_t */

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, illegal overlap */
    KDA_ERR_UNSUPPORTED = 2,   /* dk/dv other than 128, unknown dtype, device not sm_103 */
    KDA_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute, ...) */
    KDA_ERR_WORKSPACE = 4      /* workspace smaller than kda_prefill_workspace_bytes() */
} kda_status;

typedef enum {
    KDA_DTYPE_BF16 = 0,
    KDA_DTYPE_F32 = 1
} kda_dtype;

/* Bits OR-ed into *device_status by the kernels. */
#define KDA_DEV_BAD_CU_SEQLENS 0x1  /* cu_seqlens not 0 .. total_tokens non-decreasing */
#define KDA_DEV_BAD_SLOT 0x2        /* state_indices entry outside [0, num_slots) */
#define KDA_DEV_TIMEOUT 0x4         /* an on-chip wait hit its iteration limit */
#define KDA_DEV_BAD_SNAPSHOT 0x8    /* kda_prefill_snapshots: a (sequence, position) entry is invalid */
#define KDA_DEV_BOUNDS 0x10         /* only in a library built with KDA_DEBUG_BOUNDS: a kernel derived a
                                       sequence, chunk, token or snapshot range outside its buffer and
                                       skipped that work (never set by a release build) */

/*
 * Fused prologue / epilogue (kda_prefill_ex, kda_decode_step_ex,
 * kda_decode_multi_ex): the elementwise steps around the recurrence that
 * "kimi delta attn from first principles" (aryagxr) lists -- q and k
 * L2-normalised ("KDA Architecture"),
 * the update gate beta as a sigmoid of its projection, and the output gate
 * (RMSNorm of o_t, then an elementwise product with g_t) ("KDA has three
 * gates").  The prologue runs inside the kernels (pass 1 of the prefill, the
 * decode kernels); the output gate runs inside the decode kernels and, for
 * the prefill, as one pass over o and the gate after the scan (the row's
 * mean square is taken from the row it scales).
 *
 *   KDA_FUSE_L2NORM_QK   q, k <- x / sqrt(sum_c x_c^2 + l2_eps), per (token, head)
 *   KDA_FUSE_BETA_SIGMOID  beta holds logits b; beta = 1 / (1 + exp(-b)) is used
 *   KDA_FUSE_OUT_GATE    the output is y = o / sqrt(mean_c o_c^2 + rms_eps)
 *                        * rms_weight * out_gate instead of o
 *
 * rms_weight: [dv] fp32 device (NULL = all ones); out_gate: [tokens, H, dv]
 * in qkv_dtype, device, 16-byte aligned (required with KDA_FUSE_OUT_GATE
 * unless tokens = 0; tokens = total_tokens for prefill, N for a decode step,
 * N x T for kda_decode_multi_ex).  l2_eps, rms_eps >= 0.
 * The state and S_final are those of the normalised q, k and sigmoid beta.
 */
#define KDA_FUSE_L2NORM_QK 0x1u
#define KDA_FUSE_BETA_SIGMOID 0x2u
#define KDA_FUSE_OUT_GATE 0x4u
typedef struct {
    uint32_t flags;
    float l2_eps;
    float rms_eps;
    const float *rms_weight;
    const void *out_gate;
} kda_fusion;

/* Version of this header the library was built from. */
KDA_API int32_t kda_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
KDA_API const char *kda_status_string(kda_status s);

/*
 * Workspace (device bytes, 256-byte aligned start) for kda_prefill's
 * two-pass path (the fast one): the sequence schedule, the chunk table, bf16
 * copies of q, k, v when qkv_dtype is KDA_DTYPE_F32, 67,072 bytes per
 * (chunk, head) of prepared operands, counting ceil(total_tokens/64) +
 * num_seqs chunks -- about 1.05 KB per token and head -- and one fp32 state
 * per (sequence, head), 64 KB each, that carries the state between the scan's
 * pieces when the call passes no S_final.  Returns 0 for invalid arguments.
 */
KDA_API size_t kda_prefill_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs,
                                   int64_t total_tokens, int32_t H,
                                   int32_t dk, int32_t dv);

/*
 * Smallest workspace kda_prefill accepts: the schedule (+ bf16 copies for
 * fp32 inputs).  With less than kda_prefill_workspace_bytes() it runs the
 * single-pass path, one CTA per (sequence, head), which is slower for few
 * long sequences.  Returns 0 for invalid arguments.
 */
KDA_API size_t kda_prefill_min_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs,
                                       int64_t total_tokens, int32_t H,
                                       int32_t dk, int32_t dv);

/*
 * kda_prefill -- chunkwise-parallel prefill over packed variable-length
 * sequences ("Understanding Kimi Delta Attention" (pyshine), section
 * "The Chunkwise DPLR Algorithm": fixed-size chunks, exactly equivalent to
 * the sequential recurrence).  Chunk size 64, fp32 state, bf16 tensor-core
 * operands with fp32 accumulation.
 *
 *   q, k       [total_tokens, H, dk]  qkv_dtype
 *   v          [total_tokens, H, dv]  qkv_dtype
 *   log_alpha  [total_tokens, H, dk]  fp32   (per key channel; see below)
 *   beta       [total_tokens, H]      fp32
 *   S0         [num_seqs, H, dk, dv]  fp32, or NULL for zero start states
 *   cu_seqlens [num_seqs + 1]         int32, device; 0 = c_0 <= ... <= c_N = total_tokens
 *   o          [total_tokens, H, dv]  qkv_dtype (out)
 *   S_final    [num_seqs, H, dk, dv]  fp32 (out), or NULL
 *   workspace  device scratch: >= kda_prefill_workspace_bytes(...) bytes
 *              selects the two-pass path (chunk preparation for all
 *              (chunk, head) pairs in parallel, then a scan over chunks per
 *              (sequence, head, 64-column slice of dv)); >=
 *              kda_prefill_min_workspace_bytes(...) selects the single-pass
 *              path; less returns KDA_ERR_WORKSPACE.  Both paths compute the
 *              same chunk algebra.
 *
 * Sequence n covers tokens [cu_seqlens[n], cu_seqlens[n+1]) and starts from
 * S0[n] (the prefix-cache state of "Kimi Delta Attention (KDA)"
 * (codewithdark), section "KV Caching Challenges & vLLM Contribution");
 * S_final[n] is its state after the last token (S0[n] for an empty
 * sequence).  S_final may alias S0 exactly; any other overlap between an
 * output and another buffer returns KDA_ERR_INVALID_ARG.  A malformed
 * cu_seqlens sets KDA_DEV_BAD_CU_SEQLENS; the single-pass path then skips the
 * sequences whose bounds are invalid, the two-pass path writes nothing.
 *
 * Range: the chunk factorisation takes exp(+-(g_r - g_ref)) of the
 * cumulative log-decay within a chunk, so log_alpha must be >= -2.5 per step
 * (documented precondition; values below it can overflow to inf/NaN).
 * q, k, v given as fp32 are rounded to bf16 operands.
 */
KDA_API kda_status kda_prefill(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                       const float *log_alpha, const float *beta, const float *S0,
                       const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                       int32_t H, int32_t dk, int32_t dv, void *o, float *S_final,
                       void *workspace, size_t workspace_bytes, int32_t *device_status,
                       kda_stream_t stream);

/*
 * kda_prefill_snapshots -- kda_prefill that also records the state at
 * caller-chosen positions inside the sequences: the prefix-cache boundaries
 * of "Kimi Delta Attention (KDA)" (codewithdark), section "KV Caching
 * Challenges & vLLM Contribution", where a cached prefix is resumed from its
 * state instead of being recomputed.
 *
 *   snap_seq   [num_snaps] int32, device: sequence index of each entry
 *   snap_pos   [num_snaps] int32, device: tokens of that sequence consumed,
 *              a multiple of 64 or the sequence length, 0 < pos <= length
 *   S_snap     [num_snaps, H, dk, dv] fp32 (out): entry i receives the
 *              state after the first snap_pos[i] tokens of sequence
 *              snap_seq[i] -- exactly the S_final a kda_prefill over that
 *              prefix alone would return
 *
 * Entries must be sorted by (sequence, position) with no repeats.  An entry
 * that breaks a rule sets KDA_DEV_BAD_SNAPSHOT; its S_snap slice may then be
 * left unwritten (never a write outside S_snap).  All other arguments and
 * errors are those of kda_prefill; snapshots need the two-pass workspace
 * (>= kda_prefill_workspace_bytes), else KDA_ERR_WORKSPACE.
 */
KDA_API kda_status kda_prefill_snapshots(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                 const float *log_alpha, const float *beta, const float *S0,
                                 const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                 int32_t H, int32_t dk, int32_t dv, void *o, float *S_final,
                                 const int32_t *snap_seq, const int32_t *snap_pos, int32_t num_snaps,
                                 float *S_snap, void *workspace, size_t workspace_bytes,
                                 int32_t *device_status, kda_stream_t stream);

/*
 * kda_prefill_ex -- kda_prefill with the fused prologue / epilogue of
 * `fusion` (host pointer; NULL or flags = 0 is kda_prefill).  With any flag
 * set the two-pass workspace is required (>= kda_prefill_workspace_bytes),
 * else KDA_ERR_WORKSPACE.  Unknown flags, a missing out_gate, or a negative
 * eps return KDA_ERR_INVALID_ARG; out_gate overlapping o returns it too.
 */
KDA_API kda_status kda_prefill_ex(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                          const float *log_alpha, const float *beta, const float *S0,
                          const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                          int32_t H, int32_t dk, int32_t dv, void *o, float *S_final,
                          const kda_fusion *fusion, void *workspace, size_t workspace_bytes,
                          int32_t *device_status, kda_stream_t stream);

/*
 * kda_prefill_backward -- reverse-mode gradient of kda_prefill (plain
 * inputs; no fusion) for the scalar loss
 *     L = sum_{t,h,j} o[t,h,j] grad_o[t,h,j] + sum_{n,h,i,j} S_final grad_S_final,
 * i.e. the vector-Jacobian product of the recurrence of "Understanding Kimi
 * Delta Attention" (pyshine), section "The KDA Recurrence", read in the
 * erase-then-write order of "kimi delta attn from first principles"
 * (aryagxr), section "KDA".  The pages train the layer but print no
 * backward; this is the exact derivative of that update, per token.
 *
 *   q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
 *   dk, dv     the forward's inputs, as kda_prefill (S0 may be NULL = zeros)
 *   grad_o        [total_tokens, H, dv] qkv_dtype, device (dL/do)
 *   grad_S_final  [num_seqs, H, dk, dv] fp32 device, or NULL (zeros)
 *   grad_q, grad_k, grad_v, grad_log_alpha  [total_tokens, H, 128] fp32 out
 *   grad_beta     [total_tokens, H] fp32 out
 *   grad_S0       [num_seqs, H, dk, dv] fp32 out, or NULL (not computed)
 *
 * The library reruns the chunkwise forward inside the call, recording the
 * state after every 64-token chunk, then computes the gradient chunkwise in
 * fp32: one walk of the state's adjoint back over the chunks of each
 * (sequence, head), and dense per-chunk products for everything else.  The
 * gradients are those of the fp32 recurrence on the given inputs; the only
 * bf16 step is the chunkwise forward that supplies the chunk-start states.
 * Results are bitwise repeatable.
 *
 * Workspace: >= kda_prefill_backward_workspace_bytes(...) device bytes,
 * 256-byte aligned (KDA_ERR_WORKSPACE below it).  Pointers: 16-byte aligned
 * (beta, grad_beta: 4).  The outputs overlap nothing: not each other, the
 * inputs or the workspace (KDA_ERR_INVALID_ARG).  Other errors are
 * kda_prefill's; a malformed cu_seqlens sets KDA_DEV_BAD_CU_SEQLENS and leaves
 * the gradients unspecified.  Asynchronous on `stream`.
 */
KDA_API size_t kda_prefill_backward_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs, int64_t total_tokens,
                                                    int32_t H, int32_t dk, int32_t dv);
KDA_API kda_status kda_prefill_backward(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                        const float *log_alpha, const float *beta, const float *S0,
                                        const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                        int32_t H, int32_t dk, int32_t dv, const void *grad_o,
                                        const float *grad_S_final, float *grad_q, float *grad_k, float *grad_v,
                                        float *grad_log_alpha, float *grad_beta, float *grad_S0,
                                        void *workspace, size_t workspace_bytes, int32_t *device_status,
                                        kda_stream_t stream);

/*
 * kda_prefill_backward_ex -- kda_prefill_backward through the fused prologue
 * of kda_prefill_ex: q, k are the raw projections (L2-normalised per (token,
 * head) with KDA_FUSE_L2NORM_QK, "KDA Architecture") and beta the logits
 * (KDA_FUSE_BETA_SIGMOID, "KDA has three gates").  grad_q, grad_k, grad_beta
 * are then the gradients with respect to those raw inputs:
 *     dx = (dx_hat - x_hat <x_hat, dx_hat>) / sqrt(|x|^2 + l2_eps),
 *     db = dbeta_hat sigma(b) (1 - sigma(b)),
 * the exact chain rule through the prologue, taken in fp32.  The call
 * writes the normalised q, k (in qkv_dtype) and sigmoid beta into the
 * workspace, runs the plain backward on them, and applies the chain rule in
 * place.  KDA_FUSE_OUT_GATE returns KDA_ERR_UNSUPPORTED (the output gate's
 * backward needs two more outputs: kda_prefill_backward_gated); fusion NULL
 * or flags 0 is kda_prefill_backward.
 *
 * Workspace: >= kda_prefill_backward_ex_workspace_bytes(...) (the plain
 * figure plus (2 x 128 x sizeof(qkv_dtype) + 12) bytes per (token, head)).
 * Other arguments, errors and overlap rules as kda_prefill_backward.
 */
KDA_API size_t kda_prefill_backward_ex_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs,
                                                       int64_t total_tokens, int32_t H, int32_t dk, int32_t dv);
KDA_API kda_status kda_prefill_backward_ex(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                           const float *log_alpha, const float *beta, const float *S0,
                                           const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                           int32_t H, int32_t dk, int32_t dv, const void *grad_o,
                                           const float *grad_S_final, float *grad_q, float *grad_k,
                                           float *grad_v, float *grad_log_alpha, float *grad_beta,
                                           float *grad_S0, const kda_fusion *fusion, void *workspace,
                                           size_t workspace_bytes, int32_t *device_status, kda_stream_t stream);

/*
 * kda_prefill_backward_gated -- kda_prefill_backward_ex for the layer output
 * y = o / sqrt(mean_c o_c^2 + rms_eps) * rms_weight * out_gate of
 * kda_prefill_ex with KDA_FUSE_OUT_GATE (the output gate of "kimi delta attn
 * from first principles" (aryagxr), section "KDA has three gates").  With
 * r = (sum_c o_c^2 / 128 + rms_eps)^(-1/2), w = rms_weight, g = out_gate and
 * dy = grad_y = dL/dy per (token, head) row:
 *     dL/do_c = r w_c g_c dy_c - (r^3 o_c / 128) sum_j dy_j o_j w_j g_j
 *     grad_out_gate_c  = dy_c o_c r w_c
 *     grad_rms_weight_c = sum over all (token, head) rows of dy_c o_c r g_c
 * and dL/do feeds the chunkwise backward in place of grad_o.  The o here is
 * the chunkwise forward's own (rerun inside the call, rounded to qkv_dtype
 * as kda_prefill_ex would output it); dL/do is rounded to qkv_dtype, as
 * grad_o is given to kda_prefill_backward.
 *
 *   grad_y           [total_tokens, H, dv] qkv_dtype device (dL/dy)
 *   grad_out_gate    [total_tokens, H, dv] fp32 out, 16-byte aligned
 *   grad_rms_weight  [dv] fp32 out, or NULL (not computed); summed over
 *                    rows in a fixed order (bitwise repeatable)
 *   fusion           required, with KDA_FUSE_OUT_GATE set (else
 *                    KDA_ERR_INVALID_ARG) and out_gate, rms_weight, rms_eps
 *                    as given to the forward; KDA_FUSE_L2NORM_QK and
 *                    KDA_FUSE_BETA_SIGMOID act as in kda_prefill_backward_ex.
 *
 * Workspace: >= kda_prefill_backward_gated_workspace_bytes(...) (the _ex
 * figure rounded up to 256 bytes, plus 592 x 128 x 4 bytes of partial sums).
 * grad_out_gate and grad_rms_weight overlap nothing (KDA_ERR_INVALID_ARG).
 * Other arguments, errors and overlap rules as kda_prefill_backward_ex.
 */
KDA_API size_t kda_prefill_backward_gated_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs,
                                                          int64_t total_tokens, int32_t H, int32_t dk, int32_t dv);
KDA_API kda_status kda_prefill_backward_gated(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                              const float *log_alpha, const float *beta, const float *S0,
                                              const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                              int32_t H, int32_t dk, int32_t dv, const void *grad_y,
                                              const float *grad_S_final, float *grad_q, float *grad_k,
                                              float *grad_v, float *grad_log_alpha, float *grad_beta,
                                              float *grad_S0, float *grad_out_gate, float *grad_rms_weight,
                                              const kda_fusion *fusion, void *workspace, size_t workspace_bytes,
                                              int32_t *device_status, kda_stream_t stream);

/*
 * kda_decode_step -- one fused recurrent step for N sequences
 * ("Understanding Kimi Delta Attention" (pyshine), section "The Chunkwise
 * DPLR Algorithm": the step-by-step "fused recurrent mode" for decode).
 * Each head's fp32 state is read once and written once, in place.
 *
 *   q, k       [N, H, dk]  qkv_dtype        v [N, H, dv] qkv_dtype
 *   log_alpha  [N, H, dk]  fp32             beta [N, H] fp32
 *   S          [num_slots, H, dk, dv] fp32, updated in place
 *   state_indices [N] int32 device, or NULL for slot = n.  Entries must be
 *              unique (duplicates race); out-of-range entries set
 *              KDA_DEV_BAD_SLOT and that sequence is skipped (its o row is
 *              left untouched).  Slots not named are never touched.
 *   o          [N, H, dv]  qkv_dtype (out)
 */
KDA_API kda_status kda_decode_step(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                           const float *log_alpha, const float *beta, float *S,
                           int32_t num_slots, const int32_t *state_indices, int32_t N,
                           int32_t H, int32_t dk, int32_t dv, void *o,
                           int32_t *device_status, kda_stream_t stream);

/*
 * kda_decode_step_ex -- kda_decode_step with the fused prologue / epilogue
 * of `fusion` (host pointer; NULL or flags = 0 is kda_decode_step).  Errors
 * as kda_prefill_ex; out_gate is [N, H, dv].
 */
KDA_API kda_status kda_decode_step_ex(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                              const float *log_alpha, const float *beta, float *S,
                              int32_t num_slots, const int32_t *state_indices, int32_t N,
                              int32_t H, int32_t dk, int32_t dv, void *o, const kda_fusion *fusion,
                              int32_t *device_status, kda_stream_t stream);

/*
 * kda_decode_multi -- T consecutive tokens per sequence in one launch: a
 * speculative-decoding verify step or a short continuation (the fused
 * recurrent mode of "Understanding Kimi Delta Attention" (pyshine), "The
 * Chunkwise DPLR Algorithm", over T steps; the speculative-decoding path of
 * its "Scaling to Kimi K3" section).  Each head's fp32 state is read once,
 * carried through the T updates on chip, and written once, in place.  The
 * per-token arithmetic is exactly kda_decode_step's.
 *
 *   q, k       [N, T, H, dk]  qkv_dtype        v [N, T, H, dv] qkv_dtype
 *   log_alpha  [N, T, H, dk]  fp32             beta [N, T, H] fp32
 *   S          [num_slots, H, dk, dv] fp32, updated in place to the state
 *              after all T tokens
 *   state_indices, device_status: as kda_decode_step
 *   o          [N, T, H, dv]  qkv_dtype (out), o[n, t] read after token t
 *   S_steps    [N, T, H, dk, dv] fp32 (out) or NULL: the state after each
 *              token, for rolling back to an accepted prefix
 * T = 0 is a no-op.
 */
KDA_API kda_status kda_decode_multi(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                    const float *log_alpha, const float *beta, float *S,
                                    int32_t num_slots, const int32_t *state_indices, int32_t N,
                                    int32_t T, int32_t H, int32_t dk, int32_t dv, void *o,
                                    float *S_steps, int32_t *device_status, kda_stream_t stream);

/*
 * kda_decode_multi_ex -- kda_decode_multi with the fused prologue / epilogue
 * of `fusion` per token (host pointer; NULL or flags = 0 is kda_decode_multi).
 * Errors as kda_prefill_ex; out_gate is [N, T, H, dv].
 */
KDA_API kda_status kda_decode_multi_ex(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                               const float *log_alpha, const float *beta, float *S,
                               int32_t num_slots, const int32_t *state_indices, int32_t N,
                               int32_t T, int32_t H, int32_t dk, int32_t dv, void *o, float *S_steps,
                               const kda_fusion *fusion, int32_t *device_status, kda_stream_t stream);

/*
 * kda_prefill_noalloc -- kda_prefill for callers that cannot allocate device
 * memory.  The sources have no counterpart to this entry point; it exists for
 * integration.  Some callers cannot hand the library a workspace: a plugin
 * that an inference engine gives only the tensors it owns, after the engine
 * has reserved all of HBM for its caches, or a latency-critical path where
 * cudaMalloc's implicit device synchronisation is not allowed.
 *
 * Same arguments and results as kda_prefill, minus the workspace.  Its
 * scratch lives in a fixed array in device global memory inside libkda:
 * KDA_NOALLOC_MAX_SEQS int32 (256 KiB), held on every GPU that loads the
 * library until the process exits.  That is passed to kda_prefill as its
 * workspace, so the single-pass path runs (the two-pass path only for inputs
 * small enough to fit).  It allocates nothing and calls no allocating
 * routine.
 *   - num_seqs > KDA_NOALLOC_MAX_SEQS returns KDA_ERR_WORKSPACE; fp32 q/k/v
 *     (which need token-sized scratch) return KDA_ERR_UNSUPPORTED.
 *   - The first call on each device looks up the array's device address
 *     (with that device current) and caches it; make that first call before
 *     any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents
 *     (each call rewrites the part it reads before reading it).  Calls whose
 *     work overlaps on the GPU -- on different streams, or from different
 *     threads -- race on it: serialise them.
 */
#define KDA_NOALLOC_MAX_SEQS 65536

KDA_API kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                       const float *log_alpha, const float *beta, const float *S0,
                                       const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                       int32_t H, int32_t dk, int32_t dv, void *o, float *S_final,
                                       int32_t *device_status, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
