"""GB300-native Kimi Delta Attention: chunkwise prefill and fused decode (libkda).

Python names mirror the C ABI in include/kda.h:
  kda_prefill, kda_prefill_snapshots, kda_prefill_ex, kda_prefill_backward, kda_prefill_backward_ex,
  kda_prefill_backward_gated, kda_decode_step, kda_decode_step_ex, kda_decode_multi, kda_decode_multi_ex,
  kda_prefill_workspace_bytes, kda_prefill_backward_workspace_bytes,
  kda_prefill_backward_ex_workspace_bytes, kda_prefill_backward_gated_workspace_bytes, kda_status_string.
The library must be built first (``__graft_entry__.build()`` or
``python -m linear_attention_chunkwise_gb300._build``); there is no fallback.
"""
from ._binding import (  # noqa: F401
    EXPORTED_SYMBOLS,
    KDA_DEV_BAD_CU_SEQLENS,
    KDA_DEV_BAD_SLOT,
    KDA_DEV_BAD_SNAPSHOT,
    KDA_DEV_BOUNDS,
    KDA_DEV_TIMEOUT,
    KDA_DTYPE_BF16,
    KDA_DTYPE_F32,
    KDA_FUSE_BETA_SIGMOID,
    KDA_FUSE_L2NORM_QK,
    KDA_FUSE_OUT_GATE,
    KDA_ERR_CUDA,
    KDA_ERR_INVALID_ARG,
    KDA_ERR_UNSUPPORTED,
    KDA_ERR_WORKSPACE,
    KDA_OK,
    Fusion,
    KdaError,
    kda_decode_multi,
    kda_decode_multi_ex,
    kda_decode_step,
    kda_decode_step_ex,
    kda_prefill,
    kda_prefill_backward,
    kda_prefill_backward_ex,
    kda_prefill_backward_ex_workspace_bytes,
    kda_prefill_backward_gated,
    kda_prefill_backward_gated_workspace_bytes,
    kda_prefill_backward_workspace_bytes,
    kda_prefill_ex,
    kda_prefill_min_workspace_bytes,
    kda_prefill_snapshots,
    kda_prefill_workspace_bytes,
    kda_status_string,
    library_path,
    load_library,
)
