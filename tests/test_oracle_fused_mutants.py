"""Plant plausible mistakes in copies of the oracle's chain rule through the fused prologue
(oracle.kda_prefill_backward_fused); each must fail its finite-difference pin.

A mutant is the function's source with one expression replaced, executed in the oracle
module's namespace (the oracle itself is untouched).
"""
import inspect

import pytest

import oracle
from tests.test_oracle_backward_pins import fused_mismatch

# (name, original text, replacement, prologue flags whose pin must catch it)
MUTANTS = [
    ("norm_backward_drops_projection",
     "dq = (dq - qh * np.sum(qh * dq, axis=-1, keepdims=True)) / nq",
     "dq = dq / nq", (True, False)),
    ("norm_backward_projects_with_q_for_k",
     "dk = (dk - kh * np.sum(kh * dk, axis=-1, keepdims=True)) / nk",
     "dk = (dk - qh * np.sum(qh * dk, axis=-1, keepdims=True)) / nk", (True, False)),
    ("norm_backward_squares_the_norm",
     "dk = (dk - kh * np.sum(kh * dk, axis=-1, keepdims=True)) / nk",
     "dk = (dk - kh * np.sum(kh * dk, axis=-1, keepdims=True)) / nk ** 2", (True, False)),
    ("sigmoid_derivative_misses_one_minus",
     "db = db * bh * (1.0 - bh)",
     "db = db * bh", (False, True)),
    ("sigmoid_derivative_at_the_logit",
     "db = db * bh * (1.0 - bh)",
     "db = db * b64 * (1.0 - b64)", (False, True)),
]


def _mutant(old, new):
    src = inspect.getsource(oracle.kda_prefill_backward_fused)
    assert src.count(old) == 1, old
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["kda_prefill_backward_fused"]


@pytest.mark.parametrize("name,old,new,flags", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, flags):
    assert fused_mismatch(_mutant(old, new), *flags) is not None, name


def test_unmutated_copy_passes():
    src = inspect.getsource(oracle.kda_prefill_backward_fused)
    assert fused_mismatch(_mutant(src.splitlines()[0], src.splitlines()[0]), True, True) is None
