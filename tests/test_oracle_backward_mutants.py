"""Plant plausible mistakes in copies of the oracle's backward; each must fail the
finite-difference pins.

Every mutant is a patched copy of oracle/kda_oracle.c compiled into a temporary
directory on the CPU (the real oracle is untouched).  Only the backward routine
is changed, so the forward in the same copy -- the source of the finite
differences -- stays correct.  A mutant is caught when some gradient entry
differs from the central difference of the loss by more than the pins'
tolerance.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests.test_oracle_backward_pins import _fd, _problem

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "kda_oracle.c")

# (name, original text, replacement) -- each anchor occurs once, inside oracle_kda_prefill_backward
MUTANTS = [
    ("dq_reads_state_before_update",
     "acc += St[(size_t)r * dv + j] * ob[j];",
     "acc += Sp[(size_t)r * dv + j] * ob[j];"),
    ("dk_drops_erase_read_term",
     "dkk[th * dk + r] += acc;",
     "dkk[th * dk + r] += 0.0 * acc;"),
    ("dbeta_sign_flipped",
     "betabar += (double)kt[r] * acc;",
     "betabar -= (double)kt[r] * acc;"),
    ("dv_sign_flipped",
     "dvv[th * dv + j] = b * acc;",
     "dvv[th * dv + j] = -b * acc;"),
    ("adjoint_not_decayed",
     "Sb[(size_t)r * dv + j] = a * Sdb[(size_t)r * dv + j];",
     "Sb[(size_t)r * dv + j] = Sdb[(size_t)r * dv + j];"),
    ("dlog_alpha_against_undecayed_state",
     "acc += Sdb[(size_t)r * dv + j] * Sd[(size_t)r * dv + j];",
     "acc += Sdb[(size_t)r * dv + j] * Sp[(size_t)r * dv + j];"),
    ("erase_adjoint_misses_beta",
     "kSb[j] = -b * acc;",
     "kSb[j] = -acc;"),
    ("output_adjoint_not_added",
     "Sb[(size_t)r * dv + j] += (double)qt[r] * ob[j];",
     "Sb[(size_t)r * dv + j] += 0.0 * ob[j];"),
]


def _caught(lib):
    x, cu, dO, dSf = _problem(1)
    g = oracle.kda_prefill_backward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], cu, x["S0"], dO, dSf,
                                    lib=lib)
    for name, grad in zip(["q", "k", "v", "log_alpha", "beta", "S0"], g):
        for idx in np.ndindex(*x[name].shape):
            h = 2.0 ** -12
            fd = (4 * _fd(x, cu, dO, dSf, name, idx, h / 2) - _fd(x, cu, dO, dSf, name, idx, h)) / 3
            if abs(grad[idx] - fd) > 1e-7 * (1 + abs(fd)):
                return f"{name}{idx}"
    return None


def test_real_backward_passes():
    assert _caught(None) is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_backward_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    start = src.index("int oracle_kda_prefill_backward(")
    assert src.count(old) == 1 and src.index(old) > start, f"anchor for {name} not found once in the backward"
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(mpath), "-o", str(so), "-lm"],
                   check=True)
    assert _caught(oracle.load_library(str(so))) is not None, f"mutant {name} passed the finite-difference pins"
