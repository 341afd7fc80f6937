"""fp64 CPU oracle for the Kimi Delta Attention recurrence (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it; it
shares no code with the CUDA path.

The arithmetic lives in ``kda_oracle.c`` (a plain token-by-token loop in
double precision, OpenMP over (sequence, head)).  This module only compiles it
with gcc and marshals numpy arrays through ctypes.

Definition followed (see the C file header for the page citations):
``S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T``,
rows of S are key channels, ``alpha_t = exp(log_alpha_t)``, and
``o_t = S_t^T q_t`` from the updated state.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libkda_oracle.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    lib.oracle_kda_prefill.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, P, P, i32]
    lib.oracle_kda_prefill.restype = ctypes.c_int
    lib.oracle_kda_decode_step.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, P, i32]
    lib.oracle_kda_decode_step.restype = ctypes.c_int
    lib.oracle_kda_prefill_backward.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, P, P, P, P, P, P, P, P, i32]
    lib.oracle_kda_prefill_backward.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = [i32]
    lib.oracle_num_threads.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads(requested: int = 0) -> int:
    return int(_load().oracle_num_threads(int(requested)))


def kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, S0=None, nthreads: int = 0, lib=None):
    """Token-loop prefill over packed sequences.

    q, k, log_alpha: [T, H, dk]; v: [T, H, dv]; beta: [T, H];
    cu_seqlens: int [N+1]; S0: [N, H, dk, dv] or None (zeros).
    Values are taken as float32 (exact for bf16 and fp32 inputs).
    Returns (o [T, H, dv] float64, S_final [N, H, dk, dv] float64).
    ``lib`` selects another compiled copy of the oracle (used by the tests
    that plant mistakes in the oracle source); default is the real one.
    """
    q, k, v, la, b = (_f32(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    assert k.shape == (T, H, dk) and la.shape == (T, H, dk)
    assert v.shape == (T, H, dv) and b.shape == (T, H)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    s0 = None if S0 is None else _f32(S0)
    if s0 is not None:
        assert s0.shape == (N, H, dk, dv)
    o = np.zeros((T, H, dv), dtype=np.float64)
    sf = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = (lib or _load()).oracle_kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(s0),
                                    _ptr(cu), N, H, dk, dv, _ptr(o), _ptr(sf), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_kda_prefill: malformed cu_seqlens or allocation failure")
    return o, sf


def kda_prefill_backward(q, k, v, log_alpha, beta, cu_seqlens, S0, dO, dS_final=None, nthreads: int = 0, lib=None):
    """Reverse-mode gradient of kda_prefill for L = <o, dO> + <S_final, dS_final>.

    Same inputs as kda_prefill plus dO [T, H, dv] and dS_final [N, H, dk, dv] (None = 0).
    Returns (dq, dk, dv, dlog_alpha, dbeta, dS0), float64, shaped like the inputs.
    """
    q, k, v, la, b = (_f32(x) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    s0 = None if S0 is None else _f32(S0)
    do = np.ascontiguousarray(np.asarray(dO, dtype=np.float64))
    dsf = None if dS_final is None else np.ascontiguousarray(np.asarray(dS_final, dtype=np.float64))
    assert do.shape == (T, H, dv)
    out = [np.zeros((T, H, dk)), np.zeros((T, H, dk)), np.zeros((T, H, dv)), np.zeros((T, H, dk)),
           np.zeros((T, H)), np.zeros((N, H, dk, dv))]
    rc = (lib or _load()).oracle_kda_prefill_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(s0), _ptr(cu), N, H, dk, dv, _ptr(do), _ptr(dsf),
        *(_ptr(x) for x in out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_kda_prefill_backward: malformed cu_seqlens or allocation failure")
    return tuple(out)


def kda_decode_step(q, k, v, log_alpha, beta, S, state_indices=None, nthreads: int = 0, lib=None):
    """One decode step, S (float64 [slots, H, dk, dv]) updated IN PLACE.

    q, k, log_alpha: [N, H, dk]; v: [N, H, dv]; beta: [N, H].
    Returns o [N, H, dv] float64.
    """
    q, k, v, la, b = (_f32(x) for x in (q, k, v, log_alpha, beta))
    N, H, dk = q.shape
    dv = v.shape[2]
    assert isinstance(S, np.ndarray) and S.dtype == np.float64 and S.flags.c_contiguous
    slots = S.shape[0]
    assert S.shape == (slots, H, dk, dv)
    idx = None if state_indices is None else np.ascontiguousarray(np.asarray(state_indices, dtype=np.int32))
    o = np.zeros((N, H, dv), dtype=np.float64)
    rc = (lib or _load()).oracle_kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(S), slots,
                                        _ptr(idx), N, H, dk, dv, _ptr(o), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_kda_decode_step: slot index out of range")
    return o


# ------------------------------------------------------------------------
# Prologue / epilogue around the recurrence (plain fp64 definitions).  From
# "kimi delta attn from first principles" (aryagxr): q and k are
# L2-normalised ("KDA Architecture"), the update gate beta is the sigmoid of
# its projection, and the output gate multiplies RMSNorm(o_t) elementwise by
# g_t ("KDA has three gates").  The pages fix no epsilon; both take one.

def l2_normalize(x, eps: float = 0.0) -> np.ndarray:
    """x / sqrt(sum_c x_c^2 + eps) over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def sigmoid(b) -> np.ndarray:
    """1 / (1 + exp(-b))."""
    b = np.asarray(b, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-b))


def rmsnorm_gate(o, g, w=None, eps: float = 0.0) -> np.ndarray:
    """o / sqrt(mean_c o_c^2 + eps) * w * g over the last axis (w = ones when None)."""
    o = np.asarray(o, dtype=np.float64)
    y = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    if w is not None:
        y = y * np.asarray(w, dtype=np.float64)
    return y * np.asarray(g, dtype=np.float64)


def kda_prefill_backward_fused(q, k, v, log_alpha, beta, cu_seqlens, S0, dO, dS_final=None, l2norm_qk=True,
                               beta_sigmoid=True, l2_eps: float = 0.0, nthreads: int = 0, lib=None):
    """Gradient of the prefill with its fused prologue: q and k L2-normalised and beta = sigmoid(logits)
    before the recurrence ("kimi delta attn from first principles" (aryagxr), "KDA Architecture" and
    "KDA has three gates").  The recurrence's gradient is kda_prefill_backward at the normalised
    inputs; the two elementwise maps are then differentiated in fp64:
      x_hat = x / n, n = sqrt(sum_c x_c^2 + eps):  dx = (dx_hat - x_hat <x_hat, dx_hat>) / n
      beta = sigmoid(b):                           db = dbeta * beta * (1 - beta)
    Returns (dq, dk, dv, dlog_alpha, dbeta_logits_or_dbeta, dS0) in float64.
    """
    q64 = np.asarray(q, dtype=np.float64)
    k64 = np.asarray(k, dtype=np.float64)
    b64 = np.asarray(beta, dtype=np.float64)
    qh = l2_normalize(q64, l2_eps) if l2norm_qk else q64
    kh = l2_normalize(k64, l2_eps) if l2norm_qk else k64
    bh = sigmoid(b64) if beta_sigmoid else b64
    dq, dk, dv, dla, db, ds0 = kda_prefill_backward(qh, kh, v, log_alpha, bh, cu_seqlens, S0, dO, dS_final,
                                                    nthreads=nthreads, lib=lib)
    if l2norm_qk:
        nq = np.sqrt(np.sum(q64 * q64, axis=-1, keepdims=True) + l2_eps)
        nk = np.sqrt(np.sum(k64 * k64, axis=-1, keepdims=True) + l2_eps)
        dq = (dq - qh * np.sum(qh * dq, axis=-1, keepdims=True)) / nq
        dk = (dk - kh * np.sum(kh * dk, axis=-1, keepdims=True)) / nk
    if beta_sigmoid:
        db = db * bh * (1.0 - bh)
    return dq, dk, dv, dla, db, ds0


def rmsnorm_gate_backward(o, g, dy, w=None, eps: float = 0.0):
    """Gradient of y = rmsnorm_gate(o, g, w, eps) for L = <y, dy> (fp64), over the last axis of n entries:
      y_j = o_j r w_j g_j,  r = (sum_k o_k^2 / n + eps)^(-1/2),  so  dr/do_m = -r^3 o_m / n  and
      do_m = r w_m g_m dy_m - (r^3 o_m / n) sum_j dy_j o_j w_j g_j
      dg_j = dy_j o_j r w_j
      dw_j = the sum over every other axis of dy_j o_j r g_j
    Returns (do, dg, dw); dw is None when w is None (w = ones)."""
    o = np.asarray(o, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    n = o.shape[-1]
    w64 = np.ones(n) if w is None else np.asarray(w, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    wgdy = w64 * g * dy
    do = r * wgdy - (r ** 3 / n) * o * np.sum(wgdy * o, axis=-1, keepdims=True)
    dg = dy * o * r * w64
    dw = None if w is None else np.sum((dy * o * r * g).reshape(-1, n), axis=0)
    return do, dg, dw


def kda_prefill_backward_gated(q, k, v, log_alpha, beta, cu_seqlens, S0, dY, dS_final, gate, rms_weight=None,
                               rms_eps: float = 0.0, l2norm_qk=False, beta_sigmoid=False, l2_eps: float = 0.0,
                               nthreads: int = 0, lib=None):
    """Gradient of the prefill whose output passes through the output gate of "kimi delta attn from first
    principles" (aryagxr), "KDA has three gates": y = rmsnorm_gate(o, gate, rms_weight, rms_eps), for
    L = <y, dY> + <S_final, dS_final>, optionally with the fused prologue of kda_prefill_backward_fused.
    The forward o is recomputed by kda_prefill (on the prologue's outputs), the gate's backward gives
    dL/do, and kda_prefill_backward_fused carries it through the recurrence.
    Returns (dq, dk, dv, dlog_alpha, dbeta, dS0, dgate, drms_weight) in float64 (drms_weight None when
    rms_weight is None)."""
    q64 = np.asarray(q, dtype=np.float64)
    k64 = np.asarray(k, dtype=np.float64)
    b64 = np.asarray(beta, dtype=np.float64)
    qh = l2_normalize(q64, l2_eps) if l2norm_qk else q64
    kh = l2_normalize(k64, l2_eps) if l2norm_qk else k64
    bh = sigmoid(b64) if beta_sigmoid else b64
    o, _ = kda_prefill(qh, kh, v, log_alpha, bh, cu_seqlens, S0, nthreads=nthreads, lib=lib)
    do, dg, dw = rmsnorm_gate_backward(o, gate, dY, rms_weight, rms_eps)
    grads = kda_prefill_backward_fused(q, k, v, log_alpha, beta, cu_seqlens, S0, do, dS_final, l2norm_qk=l2norm_qk,
                                       beta_sigmoid=beta_sigmoid, l2_eps=l2_eps, nthreads=nthreads, lib=lib)
    return tuple(grads) + (dg, dw)
