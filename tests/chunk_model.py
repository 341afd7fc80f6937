"""CPU model of the chunkwise algebra the prefill kernel implements (test aid).

This is NOT the oracle.  It restates, in numpy, the per-chunk steps of the
CUDA prefill so that the derivation can be checked against the token-loop
oracle on the CPU, and so that the effect of bf16 operand rounding can be
studied without a GPU.  It imports nothing from the library or the oracle.

Per chunk of C rows (start state S, rows past the sequence end masked to
k = q = v = 0, beta = 0, log_alpha = 0):
  g   = inclusive cumsum of log_alpha over rows          (per key channel)
  gm  = g[C/2 - 1] (reference row), gC = g[C - 1]
  Kh  = k * exp(g - gm),  Qh = q * exp(g - gm),  Kb = k * exp(gm - g)
  A   = Kh Kb^T (strict lower part used),  QK = Qh Kb^T (lower incl. diagonal)
  T   = (I + Diag(beta) A_strict)^-1,   Tb = T Diag(beta)
  [W; MW]   = [Tb; M Tb] Kh          [U0; MU0] = [Tb; M Tb] V
  Sm  = Diag(exp(gm)) S
  [U; O]    = [U0; MU0] + [-W; Qh - MW] Sm
  S  <- Diag(exp(gC)) S + Diag(exp(gC - gm)) Kb^T U
which equals the token loop exactly in exact arithmetic.
"""
from __future__ import annotations

import numpy as np

C = 64


def _bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 -> bf16 (round to nearest even) -> float64."""
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    rounding = ((b >> 16) & 1) + 0x7FFF
    b = ((b + rounding) >> 16) << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def chunk_prefill(q, k, v, log_alpha, beta, cu_seqlens, S0=None, round_bf16=False, chunk=C):
    q, k, v, la, b = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu_seqlens) - 1
    rd = _bf16 if round_bf16 else (lambda x: x)
    o = np.zeros((T, H, dv))
    Sf = np.zeros((N, H, dk, dv))
    mid = chunk // 2 - 1
    for n in range(N):
        s0, s1 = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.asarray(S0[n, h], dtype=np.float64).copy()
            for t0 in range(s0, s1, chunk):
                L = min(chunk, s1 - t0)
                kk = np.zeros((chunk, dk)); qq = np.zeros((chunk, dk)); vv = np.zeros((chunk, dv))
                ll = np.zeros((chunk, dk)); bb = np.zeros(chunk)
                kk[:L] = k[t0:t0 + L, h]; qq[:L] = q[t0:t0 + L, h]; vv[:L] = v[t0:t0 + L, h]
                ll[:L] = la[t0:t0 + L, h]; bb[:L] = b[t0:t0 + L, h]
                g = np.cumsum(ll, axis=0)
                gm, gC = g[mid], g[chunk - 1]
                E = np.exp(g - gm)
                Kh, Qh, Kb = rd(kk * E), rd(qq * E), rd(kk / E)
                A = Kh @ Kb.T
                QK = Qh @ Kb.T
                Nm = np.tril(A, -1) * bb[:, None]
                Tm = np.linalg.inv(np.eye(chunk) + Nm)
                Tb = rd(Tm * bb[None, :])
                Mm = rd(np.tril(QK))
                MTb = rd(Mm @ Tb)
                A3 = np.vstack([Tb, MTb])
                WMW = A3 @ Kh
                UO0 = A3 @ rd(vv)
                Achain = rd(np.vstack([-WMW[:chunk], Qh - WMW[chunk:]]))
                Sm = rd(np.exp(gm)[:, None] * S)
                X = UO0 + Achain @ Sm
                U = rd(X[:chunk])
                O = X[chunk:]
                S = np.exp(gC)[:, None] * S + np.exp(gC - gm)[:, None] * (Kb.T @ U)
                o[t0:t0 + L, h] = O[:L]
            Sf[n, h] = S
    return o, Sf
