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


def chunk_backward(q, k, v, log_alpha, beta, cu_seqlens, S0, dO, dS_final=None, chunk=C):
    """Chunkwise form of the prefill gradient (fp64), the algebra of the CUDA backward.

    Per chunk, walking back with X = dL/d(state after the chunk) (dS_final for the last one),
    from the chunk-start state S (recomputed forward), with g, gm, gC, Kh, Qh, Kb as in
    chunk_prefill, Eq = exp(g - gm), Eb = exp(gm - g) and
      Lm = strict lower (Kh Kb^T),  Mm = lower incl. diagonal (Qh Kb^T),
      Tb = (I + Diag(beta) Lm)^-1 Diag(beta),  Sm = Diag(exp(gm)) S,  Xc = Diag(exp(gC - gm)) X:
      U  = Tb (V - Kh Sm)                  (rows u_t = beta_t r_t of the forward)
      R  = V - Kh Sm - Lm U                (rows r_t = v_t - S'_t^T k_t)
      dY = -Tb^T (Mm^T dO + Kb Xc)         (dL/dy_t for y_t = S'_t^T k_t);  dv = -dY
      du = Mm^T dO + Lm^T dY + Kb Xc;      dbeta_t = <du_t, r_t>
      dq = Eq * (dO Sm^T + tril(dO U^T) Kb)
      dk = Eb * (triu(U dO^T) Qh + striu(U dY^T) Kh + U Xc^T) + Eq * (dY Sm^T + stril(dY U^T) Kb)
      dg = q * dq + k * (second term - first term of dk);  dg[last row] += rowsum(S_next * X)
      dlog_alpha = reverse cumsum of dg over the chunk's rows
      X <- Diag(exp(gC)) X + Diag(exp(gm)) (Qh^T dO + Kh^T dY)
    and dS0 = X after the first chunk.
    """
    q, k, v, la, b, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_alpha, beta, dO))
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu_seqlens) - 1
    mid = chunk // 2 - 1
    out = [np.zeros((T, H, dk)), np.zeros((T, H, dk)), np.zeros((T, H, dv)), np.zeros((T, H, dk)),
           np.zeros((T, H)), np.zeros((N, H, dk, dv))]
    gq, gk, gv, gla, gb, gs0 = out

    def pieces(t0, L, h):
        kk = np.zeros((chunk, dk)); qq = np.zeros((chunk, dk)); vv = np.zeros((chunk, dv))
        ll = np.zeros((chunk, dk)); bb = np.zeros(chunk); dd = np.zeros((chunk, dv))
        kk[:L] = k[t0:t0 + L, h]; qq[:L] = q[t0:t0 + L, h]; vv[:L] = v[t0:t0 + L, h]
        ll[:L] = la[t0:t0 + L, h]; bb[:L] = b[t0:t0 + L, h]; dd[:L] = do[t0:t0 + L, h]
        g = np.cumsum(ll, axis=0)
        gm, gC = g[mid], g[chunk - 1]
        Eq, Eb = np.exp(g - gm), np.exp(gm - g)
        Kh, Qh, Kb = kk * Eq, qq * Eq, kk * Eb
        Lm = np.tril(Kh @ Kb.T, -1)
        Mm = np.tril(Qh @ Kb.T)
        Tb = np.linalg.inv(np.eye(chunk) + bb[:, None] * Lm) * bb[None, :]
        return dict(k=kk, q=qq, v=vv, b=bb, dO=dd, gm=gm, gC=gC, Eq=Eq, Eb=Eb, Kh=Kh, Qh=Qh, Kb=Kb, Lm=Lm,
                    Mm=Mm, Tb=Tb)

    for n in range(N):
        s0, s1 = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        starts = list(range(s0, s1, chunk))
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.asarray(S0[n, h], dtype=np.float64).copy()
            states = []
            for t0 in starts:  # forward: the state at every chunk start, then the final state
                states.append(S)
                p = pieces(t0, min(chunk, s1 - t0), h)
                Sm = np.exp(p["gm"])[:, None] * S
                U = p["Tb"] @ (p["v"] - p["Kh"] @ Sm)
                S = np.exp(p["gC"])[:, None] * S + np.exp(p["gC"] - p["gm"])[:, None] * (p["Kb"].T @ U)
            states.append(S)
            X = np.zeros((dk, dv)) if dS_final is None else np.asarray(dS_final[n, h], dtype=np.float64).copy()
            for c in range(len(starts) - 1, -1, -1):
                t0 = starts[c]
                L = min(chunk, s1 - t0)
                p = pieces(t0, L, h)
                Sm = np.exp(p["gm"])[:, None] * states[c]
                Xc = np.exp(p["gC"] - p["gm"])[:, None] * X
                KhSm = p["Kh"] @ Sm
                U = p["Tb"] @ (p["v"] - KhSm)
                R = p["v"] - KhSm - p["Lm"] @ U
                dY = -p["Tb"].T @ (p["Mm"].T @ p["dO"] + p["Kb"] @ Xc)
                du = p["Mm"].T @ p["dO"] + p["Lm"].T @ dY + p["Kb"] @ Xc
                dQ = p["Eq"] * (p["dO"] @ Sm.T + np.tril(p["dO"] @ U.T) @ p["Kb"])
                dKa = p["Eb"] * (np.triu(U @ p["dO"].T) @ p["Qh"] + np.triu(U @ dY.T, 1) @ p["Kh"] + U @ Xc.T)
                dKb = p["Eq"] * (dY @ Sm.T + np.tril(dY @ U.T, -1) @ p["Kb"])
                dg = p["q"] * dQ + p["k"] * (dKb - dKa)
                dg[L - 1] += np.sum(states[c + 1] * X, axis=1)
                dla = np.cumsum(dg[:L][::-1], axis=0)[::-1]
                gq[t0:t0 + L, h] = dQ[:L]
                gk[t0:t0 + L, h] = (dKa + dKb)[:L]
                gv[t0:t0 + L, h] = -dY[:L]
                gla[t0:t0 + L, h] = dla
                gb[t0:t0 + L, h] = np.sum(du * R, axis=1)[:L]
                X = np.exp(p["gC"])[:, None] * X + np.exp(p["gm"])[:, None] * (p["Qh"].T @ p["dO"] + p["Kh"].T @ dY)
            gs0[n, h] = X
    return tuple(out)
