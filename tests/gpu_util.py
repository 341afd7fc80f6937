"""Helpers for the GPU parity tests: rel-L2 and oracle runs on exact input bytes."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = 1e-2  # rel-L2 bound on o and S_final (bf16 operands, fp32 state)


def rell2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / max(den, 1e-300))


def host(t: torch.Tensor | None):
    return None if t is None else t.detach().float().cpu().numpy()


def oracle_prefill_heads(p, heads_per_seq=None):
    """Run the oracle on (a subset of) heads of packed inputs `p` (synth.PrefillInputs).

    heads_per_seq: None (all heads) or list (one list of head indices per sequence).
    Returns list over sequences of (heads, o [L, nh, 128], S_final [nh, 128, 128]).
    """
    cu = p.cu_seqlens.cpu().tolist()
    H = p.q.shape[1]
    out = []
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        heads = list(range(H)) if heads_per_seq is None else list(heads_per_seq[n])
        hidx = torch.tensor(heads, dtype=torch.long, device=p.q.device)
        sl = lambda t: host(t[a:b].index_select(1, hidx))
        S0 = None if p.S0 is None else host(p.S0[n].index_select(0, hidx))[None]
        o, sf = oracle.kda_prefill(sl(p.q), sl(p.k), sl(p.v), sl(p.log_alpha), host(p.beta[a:b].index_select(1, hidx)),
                                   [0, b - a], S0)
        out.append((heads, o, sf[0]))
    return out
