"""The chunkwise algebra (tests/chunk_model.py) equals the token-loop oracle.

Checks, on the CPU, the derivation the CUDA prefill implements: exact in
fp64 (to rounding) for full chunks, ragged tails, single tokens, packed
sequences with start states and zero-length sequences; and within the 1e-2
rel-L2 budget when every tensor-core operand is rounded to bf16 as the
kernel does, on inputs with the benchmark's statistics.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_chunkwise_gb300 import synth
from tests import chunk_model
from tests.chunk_model import chunk_prefill


def rell2(x, ref):
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def _inputs(lengths, H, dtype=torch.float32, lo=-0.2, s0_std=0.02, seed=0):
    p = synth.prefill_inputs(lengths, H, 128, dtype, lo, s0_std, seed, device="cpu")
    f = lambda t: None if t is None else t.float().numpy()
    return f(p.q), f(p.k), f(p.v), f(p.log_alpha), f(p.beta), f(p.S0), p.cu_seqlens.numpy()


@pytest.mark.parametrize("lengths", [[1], [63], [64], [65], [200], [130, 0, 7, 64]])
def test_chunk_model_exact(lengths, oracle_mod):
    q, k, v, la, b, S0, cu = _inputs(lengths, 2, seed=len(lengths) * 100 + sum(lengths))
    o_ref, s_ref = oracle.kda_prefill(q, k, v, la, b, cu, S0)
    o, s = chunk_prefill(q, k, v, la, b, cu, S0)
    assert rell2(o, o_ref) < 1e-11
    assert rell2(s, s_ref) < 1e-11


def test_chunk_model_strong_decay_exact(oracle_mod):
    """log_alpha down to -2.5 per step keeps exp(+-(g - gm)) inside fp32/bf16 range."""
    q, k, v, la, b, S0, cu = _inputs([256], 1, lo=-2.5, seed=5)
    o_ref, s_ref = oracle.kda_prefill(q, k, v, la, b, cu, S0)
    o, s = chunk_prefill(q, k, v, la, b, cu, S0)
    assert rell2(o, o_ref) < 1e-10
    assert rell2(s, s_ref) < 1e-10


def test_bf16_operand_budget(oracle_mod):
    """bf16 operands everywhere the tensor cores read them stay within 1e-2 rel-L2
    over 2048 tokens of bench-like inputs (the budget the GPU parity tests use)."""
    q, k, v, la, b, S0, cu = _inputs([2048], 1, dtype=torch.bfloat16, s0_std=None, seed=11)
    o_ref, s_ref = oracle.kda_prefill(q, k, v, la, b, cu, S0)
    o, s = chunk_prefill(q, k, v, la, b, cu, S0, round_bf16=True)
    eo, es = rell2(o, o_ref), rell2(s, s_ref)
    assert eo < 1e-2 and es < 1e-2, (eo, es)


@pytest.mark.parametrize("chunk", [8, 4])
def test_chunk_backward_matches_oracle_gradient(chunk):
    """The chunkwise gradient algebra (one walk over chunks, dense products inside a chunk)
    equals the oracle's token-by-token adjoint, incl. ragged and empty sequences, dk != dv."""
    rng = np.random.default_rng(5 + chunk)
    lengths = [37, 0, 16, 5, 9]
    H, dk, dv = 2, 6, 5
    T = sum(lengths)
    f32 = lambda *s: rng.standard_normal(s).astype(np.float32)
    q, k, v = f32(T, H, dk), f32(T, H, dk) * np.float32(0.5), f32(T, H, dv)
    la = (-0.3 * rng.random((T, H, dk))).astype(np.float32)
    b = rng.random((T, H)).astype(np.float32)
    S0 = (0.3 * rng.standard_normal((len(lengths), H, dk, dv))).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    dO = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((len(lengths), H, dk, dv))
    ref = oracle.kda_prefill_backward(q, k, v, la, b, cu, S0, dO, dSf)
    got = chunk_model.chunk_backward(q, k, v, la, b, cu, S0, dO, dSf, chunk=chunk)
    for name, r, g in zip(("q", "k", "v", "log_alpha", "beta", "S0"), ref, got):
        assert np.abs(g - r).max() <= 1e-12 * (1 + np.abs(r).max()), name
