"""Pins for the oracle's reverse-mode prefill gradient (CPU).

The gradient is checked against central finite differences of the forward
oracle on tiny problems: every entry of dq, dk, dv, dlog_alpha, dbeta and dS0
for L = <o, dO> + <S_final, dS_final>.  Inputs are exactly representable
float32 values and the step h = 2^-12 keeps x +- h exact, so the differences
see only the O(h^2) truncation (Richardson-extrapolated away) and fp64
rounding.  Non-square states (dk != dv), two packed sequences and a non-zero
S0 make a transposed operand, a dropped term or a wrong sign show up.
"""
import numpy as np
import pytest

import oracle


def _problem(seed, lengths=(3, 2), H=2, dk=3, dv=2):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    q32 = lambda *s: rng.standard_normal(s).astype(np.float32)
    x = dict(q=q32(T, H, dk), k=q32(T, H, dk) * 0.6, v=q32(T, H, dv),
             log_alpha=(-0.4 * rng.random((T, H, dk))).astype(np.float32),
             beta=rng.random((T, H)).astype(np.float32),
             S0=(0.5 * rng.standard_normal((len(lengths), H, dk, dv))).astype(np.float32))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    dO = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((len(lengths), H, dk, dv))
    return x, cu, dO, dSf


def _loss(x, cu, dO, dSf):
    o, sf = oracle.kda_prefill(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], cu, x["S0"])
    return float(np.sum(o * dO) + np.sum(sf * dSf))


def _fd(x, cu, dO, dSf, name, idx, h):
    xp = {k: v.copy() for k, v in x.items()}
    xm = {k: v.copy() for k, v in x.items()}
    xp[name][idx] += np.float32(h)
    xm[name][idx] -= np.float32(h)
    return (_loss(xp, cu, dO, dSf) - _loss(xm, cu, dO, dSf)) / (2 * h)


@pytest.mark.parametrize("seed", [1, 2])
def test_backward_matches_finite_differences(seed):
    x, cu, dO, dSf = _problem(seed)
    g = oracle.kda_prefill_backward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], cu, x["S0"], dO, dSf)
    names = ["q", "k", "v", "log_alpha", "beta", "S0"]
    for name, grad in zip(names, g):
        for idx in np.ndindex(*x[name].shape):
            h = 2.0 ** -12
            # Richardson: (4 D(h/2) - D(h)) / 3 removes the h^2 term
            fd = (4 * _fd(x, cu, dO, dSf, name, idx, h / 2) - _fd(x, cu, dO, dSf, name, idx, h)) / 3
            assert abs(grad[idx] - fd) <= 1e-7 * (1 + abs(fd)), (name, idx, grad[idx], fd)


def test_backward_without_final_gradient_and_empty_sequence():
    x, cu, dO, _ = _problem(3, lengths=(4, 0, 2), H=1, dk=2, dv=3)
    g = oracle.kda_prefill_backward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], cu, x["S0"], dO, None)
    zero = np.zeros_like(x["S0"], dtype=np.float64)
    # the empty sequence passes S0 straight to S_final: with dS_final = 0 its dS0 is 0
    np.testing.assert_array_equal(g[5][1], zero[1])
    for name, grad in zip(["q", "log_alpha", "S0"], (g[0], g[3], g[5])):
        for idx in list(np.ndindex(*x[name].shape))[::3]:
            h = 2.0 ** -12
            fd = (4 * _fd(x, cu, dO, zero, name, idx, h / 2) - _fd(x, cu, dO, zero, name, idx, h)) / 3
            assert abs(grad[idx] - fd) <= 1e-7 * (1 + abs(fd)), (name, idx)


def _fused_problem(l2norm_qk, beta_sigmoid):
    """A tiny fused-prologue problem and its loss, evaluated in fp64 by the chunkwise CPU model."""
    from tests.chunk_model import chunk_prefill
    rng = np.random.default_rng(11)
    lengths = (3, 2)
    H, dk, dv, T = 2, 3, 2, 5
    x = dict(q=rng.standard_normal((T, H, dk)) * 1.7, k=rng.standard_normal((T, H, dk)) * 0.8,
             v=rng.standard_normal((T, H, dv)), log_alpha=-0.4 * rng.random((T, H, dk)),
             beta=rng.standard_normal((T, H)) * 1.5, S0=0.5 * rng.standard_normal((len(lengths), H, dk, dv)))
    if not beta_sigmoid:  # beta taken as given: keep it in (0, 1)
        x["beta"] = oracle.sigmoid(x["beta"])
    if not l2norm_qk:  # q, k taken as given: unit rows, as the plain recurrence wants
        x["q"], x["k"] = oracle.l2_normalize(x["q"], 0.0), oracle.l2_normalize(x["k"], 0.0)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    dO = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((len(lengths), H, dk, dv))
    eps = 1e-3
    nq = (lambda a: oracle.l2_normalize(a, eps)) if l2norm_qk else (lambda a: a)
    sg = oracle.sigmoid if beta_sigmoid else (lambda a: a)

    def loss(y):
        o, sf = chunk_prefill(nq(y["q"]), nq(y["k"]), y["v"], y["log_alpha"], sg(y["beta"]), cu, y["S0"], chunk=4)
        return float(np.sum(o * dO) + np.sum(sf * dSf))

    return x, cu, dO, dSf, eps, loss


def fused_mismatch(backward_fused, l2norm_qk, beta_sigmoid):
    """First gradient entry of `backward_fused` (kda_prefill_backward_fused's signature) that differs from
    the Richardson-extrapolated central difference of the loss, or None."""
    x, cu, dO, dSf, eps, loss = _fused_problem(l2norm_qk, beta_sigmoid)

    def fd(name, idx, h):
        xp = {a: b.copy() for a, b in x.items()}
        xm = {a: b.copy() for a, b in x.items()}
        xp[name][idx] += h
        xm[name][idx] -= h
        return (loss(xp) - loss(xm)) / (2 * h)

    g = backward_fused(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], cu, x["S0"], dO, dSf,
                       l2norm_qk=l2norm_qk, beta_sigmoid=beta_sigmoid, l2_eps=eps)
    for name, grad in zip(("q", "k", "v", "log_alpha", "beta", "S0"), g):
        for idx in np.ndindex(*x[name].shape):
            h = 2.0 ** -14
            ref = (4 * fd(name, idx, h / 2) - fd(name, idx, h)) / 3
            # the oracle's C routine takes its (normalised) inputs in float32: ~1e-7 relative
            if abs(grad[idx] - ref) > 2e-6 * (1 + abs(ref)):
                return f"{name}{idx}: {grad[idx]} vs {ref}"
    return None


@pytest.mark.parametrize("l2norm_qk,beta_sigmoid", [(True, True), (True, False), (False, True)])
def test_fused_prologue_backward_matches_finite_differences(l2norm_qk, beta_sigmoid):
    """kda_prefill_backward_fused (L2 norm of q, k and / or sigmoid beta before the recurrence) against
    central differences of the fused forward evaluated in fp64 (the chunkwise CPU model, exact to
    1e-12 against the oracle loop, so no fp32 rounding enters the differences)."""
    bad = fused_mismatch(oracle.kda_prefill_backward_fused, l2norm_qk, beta_sigmoid)
    assert bad is None, bad
