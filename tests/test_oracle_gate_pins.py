"""Pins for the oracle's gradient through the output gate y = RMSNorm(o) * w * g ("kimi delta attn
from first principles" (aryagxr), "KDA has three gates"), CPU only.

(1) oracle.rmsnorm_gate_backward against central differences of oracle.rmsnorm_gate on its own;
(2) oracle.kda_prefill_backward_gated, the whole chain (prologue, recurrence, gate), against central
differences of the gated forward evaluated in fp64 by the chunkwise CPU model, on every entry of every
gradient, the gate's and the RMSNorm weight's included.  test_oracle_gate_mutants.py plants mistakes
that these pins catch.
"""
import numpy as np
import pytest

import oracle


def _richardson(f, h):
    return (4 * f(h / 2) - f(h)) / 3


def gate_mismatch(backward, with_w):
    """First entry of `backward` (rmsnorm_gate_backward's signature) off the central difference, or None."""
    rng = np.random.default_rng(21)
    o = rng.standard_normal((3, 2, 5))
    g = rng.standard_normal((3, 2, 5))
    w = 1.0 + 0.5 * rng.standard_normal(5) if with_w else None
    dy = rng.standard_normal((3, 2, 5))
    eps = 1e-2
    x = {"o": o, "g": g}
    if with_w:
        x["w"] = w

    def loss(y):
        return float(np.sum(oracle.rmsnorm_gate(y["o"], y["g"], y.get("w"), eps) * dy))

    do, dg, dw = backward(o, g, dy, w, eps)
    got = {"o": do, "g": dg, "w": dw}
    for name in x:
        for idx in np.ndindex(*x[name].shape):
            def fd(h):
                xp = {a: b.copy() for a, b in x.items()}
                xm = {a: b.copy() for a, b in x.items()}
                xp[name][idx] += h
                xm[name][idx] -= h
                return (loss(xp) - loss(xm)) / (2 * h)
            ref = _richardson(fd, 2.0 ** -10)
            if got[name] is None or abs(got[name][idx] - ref) > 1e-9 * (1 + abs(ref)):
                return f"{name}{idx}: {None if got[name] is None else got[name][idx]} vs {ref}"
    return None


@pytest.mark.parametrize("with_w", [True, False])
def test_rmsnorm_gate_backward_matches_finite_differences(with_w):
    bad = gate_mismatch(oracle.rmsnorm_gate_backward, with_w)
    assert bad is None, bad


def gated_mismatch(backward_gated, l2norm_qk, beta_sigmoid):
    """First entry of `backward_gated` (kda_prefill_backward_gated's signature) off the Richardson-
    extrapolated central difference of the gated loss, or None."""
    from tests.chunk_model import chunk_prefill
    rng = np.random.default_rng(23)
    lengths = (3, 2)
    H, dk, dv, T = 2, 3, 4, 5
    x = dict(q=rng.standard_normal((T, H, dk)) * 1.3, k=rng.standard_normal((T, H, dk)) * 0.8,
             v=rng.standard_normal((T, H, dv)), log_alpha=-0.4 * rng.random((T, H, dk)),
             beta=rng.standard_normal((T, H)) * 1.5, S0=0.5 * rng.standard_normal((len(lengths), H, dk, dv)),
             g=rng.standard_normal((T, H, dv)), w=1.0 + 0.5 * rng.standard_normal(dv))
    if not beta_sigmoid:
        x["beta"] = oracle.sigmoid(x["beta"])
    if not l2norm_qk:
        x["q"], x["k"] = oracle.l2_normalize(x["q"], 0.0), oracle.l2_normalize(x["k"], 0.0)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    dY = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((len(lengths), H, dk, dv))
    l2_eps, rms_eps = 1e-3, 1e-2
    nq = (lambda a: oracle.l2_normalize(a, l2_eps)) if l2norm_qk else (lambda a: a)
    sg = oracle.sigmoid if beta_sigmoid else (lambda a: a)

    def loss(y):
        o, sf = chunk_prefill(nq(y["q"]), nq(y["k"]), y["v"], y["log_alpha"], sg(y["beta"]), cu, y["S0"], chunk=4)
        return float(np.sum(oracle.rmsnorm_gate(o, y["g"], y["w"], rms_eps) * dY) + np.sum(sf * dSf))

    got = backward_gated(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], cu, x["S0"], dY, dSf, x["g"], x["w"],
                         rms_eps=rms_eps, l2norm_qk=l2norm_qk, beta_sigmoid=beta_sigmoid, l2_eps=l2_eps)
    for name, grad in zip(("q", "k", "v", "log_alpha", "beta", "S0", "g", "w"), got):
        for idx in np.ndindex(*x[name].shape):
            def fd(h):
                xp = {a: b.copy() for a, b in x.items()}
                xm = {a: b.copy() for a, b in x.items()}
                xp[name][idx] += h
                xm[name][idx] -= h
                return (loss(xp) - loss(xm)) / (2 * h)
            ref = _richardson(fd, 2.0 ** -14)
            # the oracle's C routine takes its (normalised) inputs in float32: ~1e-7 relative
            if abs(grad[idx] - ref) > 2e-6 * (1 + abs(ref)):
                return f"{name}{idx}: {grad[idx]} vs {ref}"
    return None


@pytest.mark.parametrize("l2norm_qk,beta_sigmoid", [(False, False), (True, True)])
def test_gated_backward_matches_finite_differences(l2norm_qk, beta_sigmoid):
    bad = gated_mismatch(oracle.kda_prefill_backward_gated, l2norm_qk, beta_sigmoid)
    assert bad is None, bad
