"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins reject every one of them.  This shows the pins are strong enough to
catch a dropped term, a wrong sign, a wrong group or k index, a wrong fp16
exponent bias and a wrong row selection."""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "zero_sign": [("(qv - zv) * sv", "(qv + zv) * sv")],
    "group_index": [("int grp = k / g;", "int grp = k % (K / g);")],
    "dropped_term": [("y[c] += xv * w[c];", "y[c] += (k ? xv * w[c] : 0.0);")],
    "reversed_k": [("j->q[(size_t)k * N + n]", "j->q[(size_t)(K - 1 - k) * N + n]")],
    "exponent_bias": [("e - 25", "e - 24")],
    "row_select": [("int m = j->rows ? j->rows[r] : r;", "int m = r;")],
    "scale_of_next_col": [("double sv = oracle_half_to_double(j->s[(size_t)grp * N + n]);",
                           "double sv = oracle_half_to_double(j->s[(size_t)grp * N + (n + 1) % N]);")],
}

PINS = [
    pins.test_half_decode_all_patterns_match_numpy,
    pins.test_code_equal_zero_gives_zero,
    lambda: pins.test_single_code_closed_form(15, 0, 15.0),
    lambda: pins.test_single_code_closed_form(0, 15, -15.0),
    pins.test_one_group_constant_zero_and_scale_is_numpy_matmul,
    pins.test_grouping_runs_along_k_not_n,
    pins.test_column_sums_closed_form,
    pins.test_linearity_in_x_exact,
    pins.test_transpose_sensitivity_nonsquare,
    pins.test_handworked_example,
    pins.test_row_subset_and_thread_count_bitwise,
]


def _build_mutant(tmp_path, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, old
        src = src.replace(old, new)
    c = tmp_path / "mutant.c"
    c.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                           str(c), "-lm"])
    return str(so)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    so = _build_mutant(tmp_path, MUTANTS[name])
    saved = oracle._lib
    try:
        oracle._lib = None
        real_build = oracle.build
        oracle.build = lambda force=False: so
        oracle._load()
        failures = 0
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failures += 1
        assert failures > 0, f"mutant {name} passed every pin"
    finally:
        oracle.build = real_build
        oracle._lib = saved
