"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a worked
example in exact fractions, brute-force matrix products, closed forms of the
special cases the pages name (Gated DeltaNet, DeltaNet, plain linear
attention, identity, pure decay), the erase-then-write property of the delta
rule, and composition invariants (prefix-cache split, varlen, decode).
``test_oracle_mutants.py`` shows that plausible mistakes planted in the oracle
fail at least one of these.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(rng, T, H, dk, dv, unit_k=True, beta_range=(0.0, 1.0), lo=-0.5, s0=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    beta = rng.uniform(*beta_range, size=(T, H))
    la = rng.uniform(lo, 0.0, size=(T, H, dk))
    S0 = rng.standard_normal((1, H, dk, dv)) * 0.5 if s0 else None
    f = lambda x: None if x is None else x.astype(np.float32)
    return f(q), f(k), f(v), f(la), f(beta), f(S0)


def run(q, k, v, la, beta, S0=None, cu=None, lib=None):
    T = q.shape[0]
    cu = [0, T] if cu is None else cu
    return oracle.kda_prefill(q, k, v, la, beta, cu, S0, lib=lib)


# ---------------------------------------------------------------- pins ----

def pin_golden_d2(lib=None):
    """Hand-worked two-token example, dk = dv = 2 (tests/golden/kda_d2_worked.json)."""
    with open(os.path.join(GOLDEN, "kda_d2_worked.json")) as fh:
        g = json.load(fh)
    toks = g["tokens"]
    q = np.array([[t["q"]] for t in toks], dtype=np.float32)
    k = np.array([[t["k"]] for t in toks], dtype=np.float32)
    v = np.array([[t["v"]] for t in toks], dtype=np.float32)
    beta = np.array([[t["beta"]] for t in toks], dtype=np.float32)
    la = np.log(np.array([[t["alpha"]] for t in toks], dtype=np.float64)).astype(np.float32)
    S0 = np.array(g["S0"], dtype=np.float32)[None, None]
    o, sf = run(q, k, v, la, beta, S0, lib=lib)
    exp_o = np.array([[float(Fraction(x)) for x in row] for row in g["expected_fractions"]["o"]])
    exp_s = np.array([[float(Fraction(x)) for x in row] for row in g["expected_fractions"]["S_final"]])
    np.testing.assert_allclose(o[:, 0, :], exp_o, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(sf[0, 0], exp_s, rtol=1e-6, atol=1e-6)


def pin_bruteforce(lib=None, seed=1):
    """S_T = A_T...A_1 S_0 + sum_i A_T...A_{i+1} beta_i k_i v_i^T, A_t = (I - beta k k^T) Diag(alpha),
    evaluated as explicit dk x dk matrix products, for T <= 8 and several (dk, dv)."""
    rng = np.random.default_rng(seed)
    for (T, dk, dv) in [(1, 4, 4), (3, 4, 3), (8, 16, 16), (5, 5, 7), (8, 128, 128)]:
        q, k, v, la, beta, S0 = rand_case(rng, T, 1, dk, dv, unit_k=False)
        o, sf = run(q, k, v, la, beta, S0, lib=lib)
        qd, kd, vd, lad, bd = (x.astype(np.float64)[:, 0] for x in (q, k, v, la, beta))
        A = [(np.eye(dk) - bd[t] * np.outer(kd[t], kd[t])) @ np.diag(np.exp(lad[t])) for t in range(T)]
        W = [bd[t] * np.outer(kd[t], vd[t]) for t in range(T)]
        for t in range(T):
            P = np.eye(dk)
            St = np.zeros((dk, dv))
            for i in range(t, -1, -1):          # A_t ... A_{i+1} applied to W_i
                St += P @ W[i]
                P = P @ A[i]
            St += P @ S0[0, 0].astype(np.float64)
            np.testing.assert_allclose(o[t, 0], St.T @ qd[t], rtol=1e-10, atol=1e-10)
            if t == T - 1:
                np.testing.assert_allclose(sf[0, 0], St, rtol=1e-10, atol=1e-10)


def pin_gdn(lib=None, seed=2):
    """A channel-broadcast alpha reduces KDA to Gated DeltaNet,
    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T (page-1 GDN equation)."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 40, 16, 12
    q, k, v, _, beta, S0 = rand_case(rng, T, 1, dk, dv)
    a = rng.uniform(-0.3, 0.0, size=(T, 1, 1)).astype(np.float32)
    la = np.broadcast_to(a, (T, 1, dk)).copy()
    o, sf = run(q, k, v, la, beta, S0, lib=lib)
    S = S0[0, 0].astype(np.float64)
    for t in range(T):
        kk, vv, qq = k[t, 0].astype(np.float64), v[t, 0].astype(np.float64), q[t, 0].astype(np.float64)
        S = np.exp(np.float64(a[t, 0, 0])) * (np.eye(dk) - beta[t, 0] * np.outer(kk, kk)) @ S \
            + beta[t, 0] * np.outer(kk, vv)
        np.testing.assert_allclose(o[t, 0], S.T @ qq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(sf[0, 0], S, rtol=1e-11, atol=1e-12)


def pin_identity(lib=None, seed=3):
    """beta = 0 and alpha = 1 leave S unchanged; the read is then S0^T q_t."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 9, 8, 5
    q, k, v, _, _, S0 = rand_case(rng, T, 2, dk, dv)
    z = np.zeros((T, 2), np.float32)
    la = np.zeros((T, 2, dk), np.float32)
    o, sf = run(q, k, v, la, z, S0, lib=lib)
    np.testing.assert_array_equal(sf[0], S0[0].astype(np.float64))
    ref = np.einsum("hrj,thr->thj", S0[0].astype(np.float64), q.astype(np.float64))
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


def pin_pure_decay(lib=None, seed=4):
    """beta = 0: S_T = Diag(prod_t alpha_t) S_0, rows (key channels) scaled; dk != dv."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 17, 6, 3
    q, k, v, la, _, S0 = rand_case(rng, T, 1, dk, dv)
    o, sf = run(q, k, v, la, np.zeros((T, 1), np.float32), S0, lib=lib)
    decay = np.exp(la.astype(np.float64)[:, 0].sum(axis=0))
    np.testing.assert_allclose(sf[0, 0], decay[:, None] * S0[0, 0].astype(np.float64), rtol=1e-12)


def pin_erase_then_write(lib=None, seed=5):
    """Unit key and beta = 1: the updated state maps k_t exactly to v_t, for any alpha
    (the erase removes the old content along k_t before the write)."""
    rng = np.random.default_rng(seed)
    dk, dv, N = 16, 16, 3
    for lo in (0.0, -0.7):
        S = (rng.standard_normal((N, 1, dk, dv)) * 0.5)
        for _ in range(6):
            q, k, v, la, _, _ = rand_case(rng, N, 1, dk, dv, lo=lo)
            if lo == 0.0:
                la[:] = 0.0
            oracle.kda_decode_step(q, k, v, la, np.ones((N, 1), np.float32), S, lib=lib)
            for n in range(N):
                np.testing.assert_allclose(S[n, 0].T @ k[n, 0].astype(np.float64),
                                           v[n, 0].astype(np.float64), rtol=1e-6, atol=1e-6)


def pin_linear_attention(lib=None, seed=6):
    """Orthonormal keys, alpha = 1, S0 = 0: no erase ever fires, so
    o_t = sum_{i<=t} beta_i (q_t . k_i) v_i (linear attention with a learning rate)."""
    rng = np.random.default_rng(seed)
    dk, dv, T = 128, 64, 100
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :T].T.astype(np.float32)[:, None, :]
    q = rng.standard_normal((T, 1, dk)).astype(np.float32)
    v = rng.standard_normal((T, 1, dv)).astype(np.float32)
    beta = rng.uniform(0, 1, (T, 1)).astype(np.float32)
    la = np.zeros((T, 1, dk), np.float32)
    o, _ = run(q, k, v, la, beta, None, lib=lib)
    kd, qd, vd, bd = (x.astype(np.float64)[:, 0] for x in (k, q, v, beta))
    scores = np.tril(qd @ kd.T) * bd[None, :]
    # float32 keys are orthonormal only to ~1e-7, so the erase terms are ~1e-7, not 0
    np.testing.assert_allclose(o[:, 0], scores @ vd, rtol=1e-5, atol=1e-5)


def pin_deltanet(lib=None, seed=7):
    """alpha = 1: the DeltaNet error-correction form S_t = S_{t-1} + beta k (v - S_{t-1}^T k)^T."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 30, 12, 9
    q, k, v, _, beta, S0 = rand_case(rng, T, 1, dk, dv, unit_k=False)
    la = np.zeros((T, 1, dk), np.float32)
    o, sf = run(q, k, v, la, beta, S0, lib=lib)
    S = S0[0, 0].astype(np.float64)
    for t in range(T):
        kk, vv, qq = (x[t, 0].astype(np.float64) for x in (k, v, q))
        S = S + beta[t, 0] * np.outer(kk, vv - S.T @ kk)
        np.testing.assert_allclose(o[t, 0], S.T @ qq, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(sf[0, 0], S, rtol=1e-10, atol=1e-10)


def pin_single_token(lib=None, seed=8):
    """From S0 = 0 one token gives S_1 = beta k v^T and o_1 = beta (q . k) v."""
    rng = np.random.default_rng(seed)
    q, k, v, la, beta, _ = rand_case(rng, 1, 3, 10, 7, unit_k=False)
    o, sf = run(q, k, v, la, beta, None, lib=lib)
    for h in range(3):
        kk, vv, qq = (x[0, h].astype(np.float64) for x in (k, v, q))
        np.testing.assert_allclose(sf[0, h], beta[0, h] * np.outer(kk, vv), rtol=1e-12)
        np.testing.assert_allclose(o[0, h], beta[0, h] * (qq @ kk) * vv, rtol=1e-12, atol=1e-14)


def pin_split_and_varlen(lib=None, seed=9):
    """Prefix-cache split: prefill(A||B) == prefill(B, S0 = S_final(A)); a packed
    batch equals its sequences run one by one; a zero-length sequence returns S0."""
    rng = np.random.default_rng(seed)
    T, H, dk, dv = 50, 2, 8, 8
    q, k, v, la, beta, S0 = rand_case(rng, T, H, dk, dv)
    o, sf = run(q, k, v, la, beta, S0, lib=lib)
    c = 23
    oa, sa = run(q[:c], k[:c], v[:c], la[:c], beta[:c], S0, lib=lib)
    ob, sb = run(q[c:], k[c:], v[c:], la[c:], beta[c:], sa.astype(np.float32), lib=lib)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(sb, sf, rtol=1e-6, atol=1e-6)
    # packed: lengths 10, 0, 25, 15 with distinct start states
    lens = [10, 0, 25, 15]
    cu = np.cumsum([0] + lens)
    S0s = (rng.standard_normal((len(lens), H, dk, dv)) * 0.3).astype(np.float32)
    op, sp = oracle.kda_prefill(q, k, v, la, beta, cu, S0s, lib=lib)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, sn = run(q[a:b], k[a:b], v[a:b], la[a:b], beta[a:b], S0s[n:n + 1], lib=lib)
        np.testing.assert_array_equal(op[a:b], on)
        np.testing.assert_array_equal(sp[n], sn[0])
    np.testing.assert_array_equal(sp[1], S0s[1].astype(np.float64))


def pin_decode_equals_prefill(lib=None, seed=10):
    """n decode steps on one state equal a prefill over the same n tokens (one function,
    two execution modes); state_indices route each sequence to its slot."""
    rng = np.random.default_rng(seed)
    T, H, dk, dv, N = 7, 2, 8, 6, 3
    slots = 5
    idx = np.array([4, 0, 2], np.int32)
    S = rng.standard_normal((slots, H, dk, dv)) * 0.3
    S_before = S.copy()
    per_seq = [rand_case(rng, T, H, dk, dv) for _ in range(N)]
    outs = []
    for t in range(T):
        qs = np.stack([c[0][t] for c in per_seq]); ks = np.stack([c[1][t] for c in per_seq])
        vs = np.stack([c[2][t] for c in per_seq]); las = np.stack([c[3][t] for c in per_seq])
        bs = np.stack([c[4][t] for c in per_seq])
        outs.append(oracle.kda_decode_step(qs, ks, vs, las, bs, S, idx, lib=lib))
    for n in range(N):
        q, k, v, la, beta, _ = per_seq[n]
        o, sf = run(q, k, v, la, beta, S_before[idx[n]][None].astype(np.float32), lib=lib)
        # S_before rounded to float32 for the prefill start state: compare loosely
        np.testing.assert_allclose(np.stack([outs[t][n] for t in range(T)]), o, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(S[idx[n]], sf[0], rtol=1e-5, atol=1e-6)
    for s in (1, 3):   # slots not named are untouched
        np.testing.assert_array_equal(S[s], S_before[s])


def pin_norm_bound(lib=None, seed=11):
    """For |k| = 1, beta in [0, 1], alpha <= 1: ||S_t||_2 <= ||S_{t-1}||_2 + beta |v|
    ((I - beta k k^T) and Diag(alpha) are contractions)."""
    rng = np.random.default_rng(seed)
    dk, dv = 16, 16
    S = rng.standard_normal((1, 1, dk, dv))
    for _ in range(40):
        q, k, v, la, beta, _ = rand_case(rng, 1, 1, dk, dv)
        prev = np.linalg.norm(S[0, 0], 2)
        oracle.kda_decode_step(q, k, v, la, beta, S, lib=lib)
        assert np.linalg.norm(S[0, 0], 2) <= prev + beta[0, 0] * np.linalg.norm(v[0, 0]) + 1e-9


PINS = [pin_golden_d2, pin_bruteforce, pin_gdn, pin_identity, pin_pure_decay, pin_erase_then_write,
        pin_linear_attention, pin_deltanet, pin_single_token, pin_split_and_varlen,
        pin_decode_equals_prefill, pin_norm_bound]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_mod):
    pin()


def test_malformed_inputs_rejected(oracle_mod):
    q = np.zeros((4, 1, 4), np.float32)
    b = np.zeros((4, 1), np.float32)
    with pytest.raises(ValueError):
        oracle.kda_prefill(q, q, q, q, b, [0, 3, 2])      # decreasing cu_seqlens
    with pytest.raises(ValueError):
        oracle.kda_decode_step(q, q, q, q, b, np.zeros((2, 1, 4, 4)), np.array([0, 1, 2, 0], np.int32))
