"""Planted mistakes in copies of the oracle must each fail some pin (CPU).

Each mutant is the oracle's C source with one plausible slip (a dropped term,
a wrong sign, a wrong index, a transposed operand, a lost scale), compiled
into a temporary library.  The committed oracle is never modified.  All
mutated indices stay inside the arrays for the pins' shapes.
"""
import os

import pytest

import oracle
from tests.test_oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "lora_oracle.c")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("y_drops_lowrank", "return base + s * low;\n}\n\nstatic double dx_elem",
     "return base;\n}\n\nstatic double dx_elem"),
    ("y_wrong_sign", "return base + s * low;\n}\n\nstatic double dx_elem",
     "return base - s * low;\n}\n\nstatic double dx_elem"),
    ("dx_drops_lowrank", "return base + s * low;\n}\n\nstatic double da_elem",
     "return base;\n}\n\nstatic double da_elem"),
    ("dx_no_scale", "return base + s * low;\n}\n\nstatic double da_elem",
     "return base + low;\n}\n\nstatic double da_elem"),
    ("da_no_scale", "    return s * acc;\n}\n\nstatic double db_elem",
     "    return acc;\n}\n\nstatic double db_elem"),
    ("db_no_scale", "return s * acc;\n}\n\n/* ---- full",
     "return acc;\n}\n\n/* ---- full"),
    ("h_wrong_index", "acc += X[m * d_in + k] * A[i * d_in + k];",
     "acc += X[m * d_in + k] * A[i * d_in + (d_in - 1 - k)];"),
    ("g_wrong_index", "acc += dY[m * d_out + o] * B[o * r + i];",
     "acc += dY[m * d_out + o] * B[(d_out - 1 - o) * r + i];"),
    ("y_base_wrong_index", "base += X[m * d_in + k] * W[o * d_in + k];",
     "base += X[m * d_in + k] * W[o * d_in + (d_in - 1 - k)];"),
    ("dx_w_not_transposed", "base += dY[m * d_out + o] * W[o * d_in + k];",
     "base += dY[m * d_out + o] * W[(k % d_out) * d_in + (o % d_in)];"),
    ("da_wrong_operand", "acc += G[m * r + i] * X[m * d_in + k];",
     "acc += G[m * r + i] * X[m * d_in + (k + 1) % d_in];"),
    ("db_uses_x_not_h", "acc += dY[m * d_out + o] * H[m * r + i];",
     "acc += dY[m * d_out + o] * H[m * r + 0 * i];"),
    ("y_lowrank_uses_a_index", "low += H[m * r + i] * B[o * r + i];",
     "low += H[m * r + i] * B[o * r + (r - 1 - i)];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutant_c = tmp_path / f"{name}.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    oracle.compile_library(str(mutant_c), str(so))
    lib = oracle.load(str(so))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


def test_anchors_match_committed_oracle():
    """The unmutated source passes every pin (sanity of the harness)."""
    lib = oracle.load()
    for pin in ALL_PINS:
        pin(lib)
