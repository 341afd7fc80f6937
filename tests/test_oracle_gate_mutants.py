"""Plant plausible mistakes in copies of the oracle's output-gate gradient
(oracle.rmsnorm_gate_backward, and the chain in oracle.kda_prefill_backward_gated); each must fail
a finite-difference pin of tests/test_oracle_gate_pins.py.  A mutant is the function's source with one
expression replaced, executed in the oracle module's namespace (the oracle itself is untouched)."""
import inspect

import pytest

import oracle
from tests.test_oracle_gate_pins import gate_mismatch, gated_mismatch

GATE_MUTANTS = [
    ("drops_the_norm_term", "do = r * wgdy - (r ** 3 / n) * o * np.sum(wgdy * o, axis=-1, keepdims=True)",
     "do = r * wgdy"),
    ("norm_term_with_r_not_r_cubed",
     "do = r * wgdy - (r ** 3 / n) * o * np.sum(wgdy * o, axis=-1, keepdims=True)",
     "do = r * wgdy - (r / n) * o * np.sum(wgdy * o, axis=-1, keepdims=True)"),
    ("norm_term_without_the_mean",
     "do = r * wgdy - (r ** 3 / n) * o * np.sum(wgdy * o, axis=-1, keepdims=True)",
     "do = r * wgdy - r ** 3 * o * np.sum(wgdy * o, axis=-1, keepdims=True)"),
    ("gate_gradient_misses_the_norm", "dg = dy * o * r * w64", "dg = dy * o * w64"),
    ("weight_gradient_misses_the_gate", "dw = None if w is None else np.sum((dy * o * r * g).reshape(-1, n), axis=0)",
     "dw = None if w is None else np.sum((dy * o * r).reshape(-1, n), axis=0)"),
]


def _mutant(fn, name, old, new):
    src = inspect.getsource(fn)
    assert src.count(old) == 1, old
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns[name]


@pytest.mark.parametrize("name,old,new", GATE_MUTANTS, ids=[m[0] for m in GATE_MUTANTS])
def test_gate_mutant_is_caught(name, old, new):
    assert gate_mismatch(_mutant(oracle.rmsnorm_gate_backward, "rmsnorm_gate_backward", old, new), True) is not None


def test_chain_mutant_is_caught():
    """dL/do handed to the recurrence's backward before the gate's chain rule (the raw dY)."""
    bad = _mutant(oracle.kda_prefill_backward_gated, "kda_prefill_backward_gated",
                  "grads = kda_prefill_backward_fused(q, k, v, log_alpha, beta, cu_seqlens, S0, do, dS_final,",
                  "grads = kda_prefill_backward_fused(q, k, v, log_alpha, beta, cu_seqlens, S0, dY, dS_final,")
    assert gated_mismatch(bad, False, False) is not None


def test_unmutated_copies_pass():
    fn = _mutant(oracle.rmsnorm_gate_backward, "rmsnorm_gate_backward", "dg = dy * o * r * w64", "dg = dy * o * r * w64")
    assert gate_mismatch(fn, True) is None
