"""ctypes binding of libkda (include/kda.h).  Argument marshalling only.

Every step of the computation runs in the CUDA kernels of libkda.so; this
module checks tensor dtypes/devices/shapes, allocates outputs with torch when
the caller does not pass them, and forwards raw device pointers and the
current CUDA stream.  There is no CPU fallback: if the library is missing or
a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_WORKSPACE = 4
KDA_DTYPE_BF16 = 0
KDA_DTYPE_F32 = 1
KDA_DEV_BAD_CU_SEQLENS = 0x1
KDA_DEV_BAD_SLOT = 0x2
KDA_DEV_TIMEOUT = 0x4
KDA_DEV_BAD_SNAPSHOT = 0x8
KDA_DEV_BOUNDS = 0x10  # only from a library built with KDA_DEBUG_BOUNDS
KDA_FUSE_L2NORM_QK = 0x1
KDA_FUSE_BETA_SIGMOID = 0x2
KDA_FUSE_OUT_GATE = 0x4


class _KdaFusion(ctypes.Structure):
    """Mirror of the C struct kda_fusion (include/kda.h)."""
    _fields_ = [("flags", ctypes.c_uint32), ("l2_eps", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("rms_weight", ctypes.c_void_p), ("out_gate", ctypes.c_void_p)]


class Fusion:
    """Fused prologue / epilogue of the _ex entry points.

    l2norm_qk: q, k <- x / sqrt(sum x^2 + l2_eps) per (token, head); beta_sigmoid: beta holds logits;
    out_gate: [tokens, H, 128] tensor (dtype of q) -> output y = RMSNorm(o) * rms_weight * out_gate.
    """

    def __init__(self, l2norm_qk=False, beta_sigmoid=False, l2_eps=1e-6, out_gate=None, rms_weight=None,
                 rms_eps=1e-6):
        self.l2norm_qk, self.beta_sigmoid, self.l2_eps = l2norm_qk, beta_sigmoid, l2_eps
        self.out_gate, self.rms_weight, self.rms_eps = out_gate, rms_weight, rms_eps

    def c_struct(self):
        flags = (KDA_FUSE_L2NORM_QK if self.l2norm_qk else 0) | (KDA_FUSE_BETA_SIGMOID if self.beta_sigmoid else 0)
        if self.out_gate is not None:
            flags |= KDA_FUSE_OUT_GATE
        return _KdaFusion(flags, float(self.l2_eps), float(self.rms_eps),
                          None if self.rms_weight is None else self.rms_weight.data_ptr(),
                          None if self.out_gate is None else self.out_gate.data_ptr())

EXPORTED_SYMBOLS = ("kda_abi_version", "kda_status_string", "kda_prefill_workspace_bytes",
                    "kda_prefill_min_workspace_bytes", "kda_prefill", "kda_decode_step", "kda_decode_multi",
                    "kda_prefill_noalloc", "kda_prefill_snapshots", "kda_prefill_ex", "kda_decode_step_ex",
                    "kda_decode_multi_ex", "kda_prefill_backward_workspace_bytes", "kda_prefill_backward",
                    "kda_prefill_backward_ex_workspace_bytes", "kda_prefill_backward_ex",
                    "kda_prefill_backward_gated_workspace_bytes", "kda_prefill_backward_gated")

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} ({status})")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Open libkda.so and declare the C signatures.  Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libkda.so is not built ({p}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(p)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lib.kda_abi_version.argtypes = []
        lib.kda_abi_version.restype = i32
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_prefill_workspace_bytes.argtypes = [ctypes.c_int, i32, i64, i32, i32, i32]
        lib.kda_prefill_workspace_bytes.restype = sz
        lib.kda_prefill_min_workspace_bytes.argtypes = [ctypes.c_int, i32, i64, i32, i32, i32]
        lib.kda_prefill_min_workspace_bytes.restype = sz
        lib.kda_prefill.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, i32, i64, i32, i32, i32, P, P, P, sz, P, P]
        lib.kda_prefill_snapshots.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, i32, i64, i32, i32, i32, P, P,
                                              P, P, i32, P, P, sz, P, P]
        lib.kda_prefill_snapshots.restype = ctypes.c_int
        FP = ctypes.POINTER(_KdaFusion)
        lib.kda_prefill_ex.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, i32, i64, i32, i32, i32, P, P, FP, P, sz,
                                       P, P]
        lib.kda_prefill_ex.restype = ctypes.c_int
        lib.kda_decode_step_ex.argtypes = [P, P, P, ctypes.c_int, P, P, P, i32, P, i32, i32, i32, i32, P, FP, P, P]
        lib.kda_decode_step_ex.restype = ctypes.c_int
        lib.kda_decode_multi_ex.argtypes = [P, P, P, ctypes.c_int, P, P, P, i32, P, i32, i32, i32, i32, i32, P, P,
                                            FP, P, P]
        lib.kda_decode_multi_ex.restype = ctypes.c_int
        lib.kda_prefill.restype = ctypes.c_int
        lib.kda_prefill_backward_workspace_bytes.argtypes = [ctypes.c_int, i32, i64, i32, i32, i32]
        lib.kda_prefill_backward_workspace_bytes.restype = sz
        lib.kda_prefill_backward.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, i32, i64, i32, i32, i32, P, P,
                                             P, P, P, P, P, P, P, sz, P, P]
        lib.kda_prefill_backward.restype = ctypes.c_int
        lib.kda_prefill_backward_ex_workspace_bytes.argtypes = [ctypes.c_int, i32, i64, i32, i32, i32]
        lib.kda_prefill_backward_ex_workspace_bytes.restype = sz
        lib.kda_prefill_backward_ex.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, i32, i64, i32, i32, i32, P, P,
                                                P, P, P, P, P, P, FP, P, sz, P, P]
        lib.kda_prefill_backward_ex.restype = ctypes.c_int
        lib.kda_prefill_backward_gated_workspace_bytes.argtypes = [ctypes.c_int, i32, i64, i32, i32, i32]
        lib.kda_prefill_backward_gated_workspace_bytes.restype = sz
        lib.kda_prefill_backward_gated.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, i32, i64, i32, i32, i32, P,
                                                   P, P, P, P, P, P, P, P, P, FP, P, sz, P, P]
        lib.kda_prefill_backward_gated.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [P, P, P, ctypes.c_int, P, P, P, i32, P, i32, i32, i32, i32, P, P, P]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_decode_multi.argtypes = [P, P, P, ctypes.c_int, P, P, P, i32, P, i32, i32, i32, i32, i32, P, P, P, P]
        lib.kda_decode_multi.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def kda_status_string(status: int) -> str:
    return load_library().kda_status_string(int(status)).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t == torch.float32:
        return KDA_DTYPE_F32
    raise TypeError(f"q/k/v dtype must be bfloat16 or float32, got {t}")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t: torch.Tensor | None, name: str, dtype=None, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def kda_prefill_workspace_bytes(qkv_dtype, num_seqs: int, total_tokens: int, H: int, dk: int = 128,
                                dv: int = 128) -> int:
    code = qkv_dtype if isinstance(qkv_dtype, int) else _dtype_code(qkv_dtype)
    return int(load_library().kda_prefill_workspace_bytes(code, int(num_seqs), int(total_tokens), int(H),
                                                          int(dk), int(dv)))


def kda_prefill_min_workspace_bytes(qkv_dtype, num_seqs: int, total_tokens: int, H: int, dk: int = 128,
                                    dv: int = 128) -> int:
    code = qkv_dtype if isinstance(qkv_dtype, int) else _dtype_code(qkv_dtype)
    return int(load_library().kda_prefill_min_workspace_bytes(code, int(num_seqs), int(total_tokens), int(H),
                                                              int(dk), int(dv)))


def kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, S0=None, *, o=None, S_final=None, return_final=True,
                workspace=None, device_status=None, stream=None, path="two_pass"):
    """Chunkwise prefill over packed sequences (see include/kda.h).

    q, k: [T, H, 128]; v: [T, H, 128] (bf16 or fp32); log_alpha: [T, H, 128] fp32;
    beta: [T, H] fp32; cu_seqlens: int32 [N+1] on the device; S0: fp32 [N, H, 128, 128] or None.
    path: "two_pass" or "single_pass" -- sizes the workspace allocated here (the library picks
    the path from the workspace size).  Returns (o, S_final) -- S_final is None when
    return_final is False and none was given.
    """
    lib = load_library()
    dev = q.device
    _check(q, "q", device=dev)
    code = _dtype_code(q.dtype)
    _check(k, "k", q.dtype, dev)
    _check(v, "v", q.dtype, dev)
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _check(S0, "S0", torch.float32, dev)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, dk]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    if N < 0:
        raise ValueError("cu_seqlens must have at least one entry")
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _check(o, "o", q.dtype, dev)
    if S_final is None and return_final:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check(S_final, "S_final", torch.float32, dev)
    if path not in ("two_pass", "single_pass"):
        raise ValueError(f"unknown prefill path {path!r}")
    query = lib.kda_prefill_workspace_bytes if path == "two_pass" else lib.kda_prefill_min_workspace_bytes
    need = int(query(code, N, T, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8, dev)
    _check(device_status, "device_status", torch.int32, dev)
    st = lib.kda_prefill(_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S0), _ptr(cu_seqlens),
                         N, T, H, dk, dv, _ptr(o), _ptr(S_final), _ptr(workspace), workspace.numel(),
                         _ptr(device_status), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError("kda_prefill", st, kda_status_string(st))
    return o, S_final


def kda_prefill_snapshots(q, k, v, log_alpha, beta, cu_seqlens, snap_seq, snap_pos, S0=None, *, o=None,
                          S_final=None, S_snap=None, workspace=None, device_status=None, stream=None):
    """kda_prefill that also returns the state at (sequence, position) entries (see include/kda.h).

    snap_seq, snap_pos: int32 [M] on the device, sorted by (sequence, position); each position is a
    multiple of 64 or the sequence length.  Returns (o, S_final, S_snap) with S_snap [M, H, 128, 128].
    """
    lib = load_library()
    dev = q.device
    _check(q, "q", device=dev)
    code = _dtype_code(q.dtype)
    for t, n, dt in ((k, "k", q.dtype), (v, "v", q.dtype), (log_alpha, "log_alpha", torch.float32),
                     (beta, "beta", torch.float32), (cu_seqlens, "cu_seqlens", torch.int32),
                     (snap_seq, "snap_seq", torch.int32), (snap_pos, "snap_pos", torch.int32),
                     (S0, "S0", torch.float32)):
        _check(t, n, dt, dev)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, dk]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    M = snap_seq.numel()
    if snap_pos.numel() != M:
        raise ValueError("snap_seq and snap_pos must have the same length")
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    if S_final is None:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if S_snap is None:
        S_snap = torch.empty((M, H, dk, dv), dtype=torch.float32, device=dev)
    for t, n in ((o, "o"), (S_final, "S_final"), (S_snap, "S_snap")):
        _check(t, n, q.dtype if n == "o" else torch.float32, dev)
    need = int(lib.kda_prefill_workspace_bytes(code, N, T, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8, dev)
    _check(device_status, "device_status", torch.int32, dev)
    st = lib.kda_prefill_snapshots(_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S0),
                                   _ptr(cu_seqlens), N, T, H, dk, dv, _ptr(o), _ptr(S_final), _ptr(snap_seq),
                                   _ptr(snap_pos), M, _ptr(S_snap), _ptr(workspace), workspace.numel(),
                                   _ptr(device_status), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError("kda_prefill_snapshots", st, kda_status_string(st))
    return o, S_final, S_snap


def kda_prefill_backward_workspace_bytes(qkv_dtype, num_seqs: int, total_tokens: int, H: int, dk: int = 128,
                                         dv: int = 128) -> int:
    code = qkv_dtype if isinstance(qkv_dtype, int) else _dtype_code(qkv_dtype)
    return int(load_library().kda_prefill_backward_workspace_bytes(code, int(num_seqs), int(total_tokens), int(H),
                                                                   int(dk), int(dv)))


def kda_prefill_backward_ex_workspace_bytes(qkv_dtype, num_seqs: int, total_tokens: int, H: int, dk: int = 128,
                                            dv: int = 128) -> int:
    code = qkv_dtype if isinstance(qkv_dtype, int) else _dtype_code(qkv_dtype)
    return int(load_library().kda_prefill_backward_ex_workspace_bytes(code, int(num_seqs), int(total_tokens),
                                                                      int(H), int(dk), int(dv)))


def kda_prefill_backward_gated_workspace_bytes(qkv_dtype, num_seqs: int, total_tokens: int, H: int,
                                               dk: int = 128, dv: int = 128) -> int:
    code = qkv_dtype if isinstance(qkv_dtype, int) else _dtype_code(qkv_dtype)
    return int(load_library().kda_prefill_backward_gated_workspace_bytes(code, int(num_seqs), int(total_tokens),
                                                                         int(H), int(dk), int(dv)))


def kda_prefill_backward(q, k, v, log_alpha, beta, cu_seqlens, grad_o, S0=None, grad_S_final=None, *,
                         need_grad_S0=True, grads=None, workspace=None, device_status=None, stream=None):
    """Gradient of kda_prefill for L = <o, grad_o> + <S_final, grad_S_final> (see include/kda.h).

    grad_o: [T, H, 128] in the dtype of q; grad_S_final: fp32 [N, H, 128, 128] or None (zeros).
    Returns (grad_q, grad_k, grad_v, grad_log_alpha, grad_beta, grad_S0), all fp32; grad_S0 is None
    when need_grad_S0 is False.  `grads` may pass those six output tensors in.
    """
    return _backward(q, k, v, log_alpha, beta, cu_seqlens, grad_o, S0, grad_S_final, need_grad_S0, grads,
                     workspace, device_status, stream, None)


def kda_prefill_backward_ex(q, k, v, log_alpha, beta, cu_seqlens, grad_o, S0=None, grad_S_final=None, *,
                            fusion=None, need_grad_S0=True, grads=None, workspace=None, device_status=None,
                            stream=None):
    """kda_prefill_backward through the fused prologue of `fusion` (a Fusion: l2norm_qk, beta_sigmoid).

    q, k are the raw projections and beta the logits, as kda_prefill_ex takes them; grad_q, grad_k,
    grad_beta are with respect to those.  An output gate raises KdaError (KDA_ERR_UNSUPPORTED).
    """
    return _backward(q, k, v, log_alpha, beta, cu_seqlens, grad_o, S0, grad_S_final, need_grad_S0, grads,
                     workspace, device_status, stream, fusion)


def kda_prefill_backward_gated(q, k, v, log_alpha, beta, cu_seqlens, grad_y, S0=None, grad_S_final=None, *,
                               fusion, need_grad_S0=True, need_grad_rms_weight=True, grads=None, workspace=None,
                               device_status=None, stream=None):
    """Gradient of kda_prefill_ex's gated output y = RMSNorm(o) * rms_weight * out_gate (see include/kda.h).

    `fusion` must carry out_gate (and rms_weight, rms_eps as given to the forward); its prologue flags act
    as in kda_prefill_backward_ex.  grad_y: [T, H, 128] in the dtype of q.  Returns (grad_q, grad_k,
    grad_v, grad_log_alpha, grad_beta, grad_S0, grad_out_gate, grad_rms_weight), all fp32; grad_S0 and
    grad_rms_weight are None when not asked for.  `grads` may pass those eight tensors in.
    """
    if fusion is None or fusion.out_gate is None:
        raise ValueError("kda_prefill_backward_gated needs a fusion with out_gate")
    return _backward(q, k, v, log_alpha, beta, cu_seqlens, grad_y, S0, grad_S_final, need_grad_S0, grads,
                     workspace, device_status, stream, fusion, gated=True, need_grad_w=need_grad_rms_weight)


def _backward(q, k, v, log_alpha, beta, cu_seqlens, grad_o, S0, grad_S_final, need_grad_S0, grads, workspace,
              device_status, stream, fusion, gated=False, need_grad_w=False):
    lib = load_library()
    dev = q.device
    _check(q, "q", device=dev)
    code = _dtype_code(q.dtype)
    for t, n, dt in ((k, "k", q.dtype), (v, "v", q.dtype), (log_alpha, "log_alpha", torch.float32),
                     (beta, "beta", torch.float32), (cu_seqlens, "cu_seqlens", torch.int32),
                     (S0, "S0", torch.float32), (grad_o, "grad_o", q.dtype),
                     (grad_S_final, "grad_S_final", torch.float32)):
        _check(t, n, dt, dev)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, dk]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    if N < 0:
        raise ValueError("cu_seqlens must have at least one entry")
    if grads is None:
        f32 = dict(dtype=torch.float32, device=dev)
        grads = (torch.empty((T, H, dk), **f32), torch.empty((T, H, dk), **f32), torch.empty((T, H, dv), **f32),
                 torch.empty((T, H, dk), **f32), torch.empty((T, H), **f32),
                 torch.empty((N, H, dk, dv), **f32) if need_grad_S0 else None)
        if gated:
            grads += (torch.empty((T, H, dv), **f32), torch.empty((dv,), **f32) if need_grad_w else None)
    names = ("grad_q", "grad_k", "grad_v", "grad_log_alpha", "grad_beta", "grad_S0") + (
        ("grad_out_gate", "grad_rms_weight") if gated else ())
    if len(grads) != len(names):
        raise ValueError(f"grads must hold {len(names)} tensors")
    for t, n in zip(grads, names):
        _check(t, n, torch.float32, dev)
    fused = fusion is not None
    query = (lib.kda_prefill_backward_gated_workspace_bytes if gated else
             lib.kda_prefill_backward_ex_workspace_bytes if fused else lib.kda_prefill_backward_workspace_bytes)
    need = int(query(code, N, T, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8, dev)
    _check(device_status, "device_status", torch.int32, dev)
    gq, gk, gv, gla, gb, gs0 = grads[:6]
    args = [_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S0), _ptr(cu_seqlens), N, T, H, dk,
            dv, _ptr(grad_o), _ptr(grad_S_final), _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gla), _ptr(gb), _ptr(gs0)]
    tail = [_ptr(workspace), workspace.numel(), _ptr(device_status), _stream_handle(stream)]
    if gated:
        name = "kda_prefill_backward_gated"
        fz = _check_fusion(fusion, q, T)
        st = lib.kda_prefill_backward_gated(*args, _ptr(grads[6]), _ptr(grads[7]), ctypes.byref(fz), *tail)
        if st != KDA_OK:
            raise KdaError(name, st, kda_status_string(st))
        return tuple(grads)
    if fused:
        name = "kda_prefill_backward_ex"
        fz = _check_fusion(fusion, q, T)
        st = lib.kda_prefill_backward_ex(*args, ctypes.byref(fz), *tail)
    else:
        name = "kda_prefill_backward"
        st = lib.kda_prefill_backward(*args, *tail)
    if st != KDA_OK:
        raise KdaError(name, st, kda_status_string(st))
    return gq, gk, gv, gla, gb, gs0


def _check_fusion(fusion, q, tokens):
    if fusion is None:
        return None
    if fusion.out_gate is not None:
        _check(fusion.out_gate, "out_gate", q.dtype, q.device)
        if tuple(fusion.out_gate.shape) != (tokens, q.shape[1], 128):
            raise ValueError("out_gate must be [tokens, H, 128]")
    if fusion.rms_weight is not None:
        _check(fusion.rms_weight, "rms_weight", torch.float32, q.device)
    return fusion.c_struct()


def kda_prefill_ex(q, k, v, log_alpha, beta, cu_seqlens, S0=None, *, fusion=None, o=None, S_final=None,
                   workspace=None, device_status=None, stream=None):
    """kda_prefill with the fused prologue / epilogue of `fusion` (a Fusion); returns (o, S_final)."""
    lib = load_library()
    dev = q.device
    _check(q, "q", device=dev)
    code = _dtype_code(q.dtype)
    for t, n, dt in ((k, "k", q.dtype), (v, "v", q.dtype), (log_alpha, "log_alpha", torch.float32),
                     (beta, "beta", torch.float32), (cu_seqlens, "cu_seqlens", torch.int32),
                     (S0, "S0", torch.float32)):
        _check(t, n, dt, dev)
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    fz = _check_fusion(fusion, q, T)
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    if S_final is None:
        S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check(o, "o", q.dtype, dev)
    _check(S_final, "S_final", torch.float32, dev)
    need = int(lib.kda_prefill_workspace_bytes(code, N, T, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8, dev)
    _check(device_status, "device_status", torch.int32, dev)
    st = lib.kda_prefill_ex(_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S0),
                            _ptr(cu_seqlens), N, T, H, dk, dv, _ptr(o), _ptr(S_final),
                            None if fz is None else ctypes.byref(fz), _ptr(workspace), workspace.numel(),
                            _ptr(device_status), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError("kda_prefill_ex", st, kda_status_string(st))
    return o, S_final


def kda_decode_step_ex(q, k, v, log_alpha, beta, S, state_indices=None, *, fusion=None, o=None,
                       device_status=None, stream=None):
    """kda_decode_step with the fused prologue / epilogue of `fusion` (a Fusion); returns o."""
    lib = load_library()
    dev = q.device
    _check(q, "q", device=dev)
    code = _dtype_code(q.dtype)
    for t, n, dt in ((k, "k", q.dtype), (v, "v", q.dtype), (log_alpha, "log_alpha", torch.float32),
                     (beta, "beta", torch.float32), (S, "S", torch.float32),
                     (state_indices, "state_indices", torch.int32)):
        _check(t, n, dt, dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    fz = _check_fusion(fusion, q, N)
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    _check(o, "o", q.dtype, dev)
    _check(device_status, "device_status", torch.int32, dev)
    st = lib.kda_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S),
                                S.shape[0], _ptr(state_indices), N, H, dk, dv, _ptr(o),
                                None if fz is None else ctypes.byref(fz), _ptr(device_status),
                                _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError("kda_decode_step_ex", st, kda_status_string(st))
    return o


def kda_decode_step(q, k, v, log_alpha, beta, S, state_indices=None, *, o=None, device_status=None, stream=None):
    """One fused decode step; S [slots, H, 128, 128] fp32 is updated in place.

    q, k, v: [N, H, 128] (bf16 or fp32); log_alpha: [N, H, 128] fp32; beta: [N, H] fp32;
    state_indices: int32 [N] or None.  Returns o [N, H, 128].
    """
    lib = load_library()
    dev = q.device
    _check(q, "q", device=dev)
    code = _dtype_code(q.dtype)
    _check(k, "k", q.dtype, dev)
    _check(v, "v", q.dtype, dev)
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(S, "S", torch.float32, dev)
    _check(state_indices, "state_indices", torch.int32, dev)
    _check(device_status, "device_status", torch.int32, dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    _check(o, "o", q.dtype, dev)
    st = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S), S.shape[0],
                             _ptr(state_indices), N, H, dk, dv, _ptr(o), _ptr(device_status),
                             _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError("kda_decode_step", st, kda_status_string(st))
    return o


def kda_decode_multi(q, k, v, log_alpha, beta, S, state_indices=None, *, o=None, S_steps=None,
                     return_steps=False, device_status=None, stream=None):
    """T tokens per sequence in one launch; S [slots, H, 128, 128] fp32 is updated in place.

    q, k, v: [N, T, H, 128] (bf16 or fp32); log_alpha: [N, T, H, 128] fp32; beta: [N, T, H] fp32;
    state_indices: int32 [N] or None.  Returns o [N, T, H, 128], or (o, S_steps) when
    return_steps (S_steps [N, T, H, 128, 128] fp32: the state after each token).
    """
    return _decode_multi(q, k, v, log_alpha, beta, S, state_indices, None, o, S_steps, return_steps,
                         device_status, stream)


def kda_decode_multi_ex(q, k, v, log_alpha, beta, S, state_indices=None, *, fusion=None, o=None, S_steps=None,
                        return_steps=False, device_status=None, stream=None):
    """kda_decode_multi with the fused prologue / epilogue of `fusion` (a Fusion; out_gate [N, T, H, 128])."""
    return _decode_multi(q, k, v, log_alpha, beta, S, state_indices, fusion, o, S_steps, return_steps,
                         device_status, stream)


def _decode_multi(q, k, v, log_alpha, beta, S, state_indices, fusion, o, S_steps, return_steps, device_status,
                  stream):
    lib = load_library()
    dev = q.device
    _check(q, "q", device=dev)
    code = _dtype_code(q.dtype)
    _check(k, "k", q.dtype, dev)
    _check(v, "v", q.dtype, dev)
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(S, "S", torch.float32, dev)
    _check(state_indices, "state_indices", torch.int32, dev)
    _check(device_status, "device_status", torch.int32, dev)
    if q.dim() != 4:
        raise ValueError("q must be [N, T, H, dk]")
    N, T, H, dk = q.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((N, T, H, dv), dtype=q.dtype, device=dev)
    _check(o, "o", q.dtype, dev)
    if S_steps is None and return_steps:
        S_steps = torch.empty((N, T, H, dk, dv), dtype=torch.float32, device=dev)
    _check(S_steps, "S_steps", torch.float32, dev)
    if fusion is None:
        st = lib.kda_decode_multi(_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S),
                                  S.shape[0], _ptr(state_indices), N, T, H, dk, dv, _ptr(o), _ptr(S_steps),
                                  _ptr(device_status), _stream_handle(stream))
        name = "kda_decode_multi"
    else:
        if fusion.out_gate is not None and tuple(fusion.out_gate.shape) != (N, T, H, dv):
            raise ValueError("out_gate must be [N, T, H, 128]")
        fz = fusion.c_struct()
        if fusion.out_gate is not None:
            _check(fusion.out_gate, "out_gate", q.dtype, dev)
        if fusion.rms_weight is not None:
            _check(fusion.rms_weight, "rms_weight", torch.float32, dev)
        st = lib.kda_decode_multi_ex(_ptr(q), _ptr(k), _ptr(v), code, _ptr(log_alpha), _ptr(beta), _ptr(S),
                                     S.shape[0], _ptr(state_indices), N, T, H, dk, dv, _ptr(o), _ptr(S_steps),
                                     ctypes.byref(fz), _ptr(device_status), _stream_handle(stream))
        name = "kda_decode_multi_ex"
    if st != KDA_OK:
        raise KdaError(name, st, kda_status_string(st))
    return (o, S_steps) if return_steps else o
