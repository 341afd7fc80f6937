"""Plant plausible mistakes in copies of the oracle source; each must fail a pin.

The real oracle is untouched: every mutant is a patched copy of
oracle/kda_oracle.c compiled into a temporary directory on the CPU.  This
shows that the pins in test_oracle_pins.py constrain the oracle's reading of
the pages (step order, decay axis, read vector, read-after-update), not only
its arithmetic.
"""
import os
import subprocess

import pytest

import oracle
from tests.test_oracle_pins import PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "kda_oracle.c")

# (name, original text, replacement)
MUTANTS = [
    ("decay_columns_not_rows",
     "Sd[(size_t)r * dv + j] = a * S[(size_t)r * dv + j];",
     "Sd[(size_t)r * dv + j] = exp((double)log_alpha[j % dk]) * S[(size_t)r * dv + j];"),
    ("erase_before_decay",
     "for (int j = 0; j < dv; ++j) kS[j] += kr * Sd[(size_t)r * dv + j];",
     "for (int j = 0; j < dv; ++j) kS[j] += kr * S[(size_t)r * dv + j];"),
    ("erase_sign_flipped",
     "- bk * kS[j] + bk * (double)v[j];",
     "+ bk * kS[j] + bk * (double)v[j];"),
    ("write_without_beta",
     "- bk * kS[j] + bk * (double)v[j];",
     "- bk * kS[j] + (double)k[r] * (double)v[j];"),
    ("gate_not_exponentiated",
     "double a = exp((double)log_alpha[r]);",
     "double a = 1.0 + (double)log_alpha[r];"),
    ("read_with_key",
     "double qr = (double)q[r];",
     "double qr = (double)k[r];"),
    ("read_before_update",
     "for (int j = 0; j < dv; ++j) o[j] += qr * S[(size_t)r * dv + j];",
     "for (int j = 0; j < dv; ++j) o[j] += qr * Sd[(size_t)r * dv + j];"),
    ("read_transposed",
     "for (int j = 0; j < dv; ++j) o[j] += qr * S[(size_t)r * dv + j];",
     "for (int j = 0; j < dv; ++j) o[j] += (double)q[j % dk] * S[(size_t)(j % dk) * dv + (r % dv)];"),
    ("decay_uses_previous_token_gate",
     "double a = exp((double)log_alpha[r]);",
     "double a = exp((double)log_alpha[r] * 0.5);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(mpath), "-o", str(so), "-lm"],
                   check=True)
    lib = oracle.load_library(str(so))
    caught = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
