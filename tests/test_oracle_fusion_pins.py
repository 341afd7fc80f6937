"""Pins for the oracle's prologue / epilogue definitions (CPU).

Each is checked against facts fixed by its definition, not a retyped formula:
unit norm and scale invariance for the L2 normalisation, the symmetry and
known values of the sigmoid, and the RMSNorm of a constant vector, unit mean
square and scale invariance for the output gate.
"""
import numpy as np

import oracle


def test_l2_normalize_unit_norm_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 3, 128))
    y = oracle.l2_normalize(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.l2_normalize(3.5 * x), y, rtol=1e-14)
    np.testing.assert_allclose(oracle.l2_normalize(np.array([3.0, 4.0])), [0.6, 0.8], rtol=1e-15)
    # eps enters under the square root: |[3, 4]|^2 + 11 = 36
    np.testing.assert_allclose(oracle.l2_normalize(np.array([3.0, 4.0]), 11.0), [0.5, 4.0 / 6.0], rtol=1e-15)


def test_sigmoid_values_and_symmetry():
    assert oracle.sigmoid(0.0) == 0.5
    np.testing.assert_allclose(oracle.sigmoid(np.log(3.0)), 0.75, rtol=1e-15)
    b = np.linspace(-8, 8, 33)
    np.testing.assert_allclose(oracle.sigmoid(-b), 1.0 - oracle.sigmoid(b), atol=1e-15)
    assert np.all(np.diff(oracle.sigmoid(b)) > 0)


def test_rmsnorm_gate_constant_vector_and_invariants():
    rng = np.random.default_rng(2)
    w = rng.standard_normal(128)
    g = rng.standard_normal(128)
    # RMSNorm of a constant vector c is sign(c) everywhere
    np.testing.assert_allclose(oracle.rmsnorm_gate(np.full(128, -2.5), g, w), -w * g, rtol=1e-14)
    o = rng.standard_normal((5, 128))
    y = oracle.rmsnorm_gate(o, np.ones(128))
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rmsnorm_gate(7.0 * o, g, w), oracle.rmsnorm_gate(o, g, w), rtol=1e-13)
    # eps: mean square 1 + eps 3 -> divide by 2
    np.testing.assert_allclose(oracle.rmsnorm_gate(np.ones(128), np.ones(128), None, 3.0), 0.5, rtol=1e-15)
