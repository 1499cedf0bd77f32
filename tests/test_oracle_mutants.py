"""Plant plausible mistakes in copies of the oracle and show the pins catch each.

Every mutant is the oracle source with one textual change, compiled to a
temporary library on the CPU.  A mutant that passes every pin would mean the
pins cannot tell that mistake from the real definition.
"""
import os
import tempfile

import pytest

import oracle.oracle as O
from tests import oracle_pins as P

SRC = os.path.join(os.path.dirname(O.__file__), "oracle.c")

MUTANTS = {
    "drop_last_k_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    "wrong_sign": ("acc += a * b;", "acc -= a * b;"),
    "s1_without_abs": ("mag += fabs(a) * fabs(b);", "mag += a * b;"),
    "fp32_accumulator": ("double acc = 0.0, mag = 0.0;", "float acc = 0.0f; double mag = 0.0;"),
    "residual_transposed": ("y += oracle_bf16_decode(res[m * N + n]);\n        if (y_ref)",
                            "y += oracle_bf16_decode(res[n * M + m]);\n        if (y_ref)"),
    "residual_dropped": ("if (res)\n            y += oracle_bf16_decode(res[m * N + n]);\n        if (y_ref)",
                         "if (0)\n            y += oracle_bf16_decode(res[m * N + n]);\n        if (y_ref)"),
    "ties_away_from_zero": ("frac > 0.5 || (frac == 0.5 && fmod(qi, 2.0) != 0.0)", "frac >= 0.5"),
    "truncate_instead_of_round": ("frac > 0.5 || (frac == 0.5 && fmod(qi, 2.0) != 0.0)", "0"),
    "ulp_off_by_one_binade": ("return ldexp(1.0, (e - 1) - 7);", "return ldexp(1.0, e - 7);"),
    "no_subnormal_range": ("if (!(a >= 0x1p-126))", "if (!(a > 0.0))"),
    "decode_shift_wrong": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "w_row_stride_off": ("oracle_point(K, x + m * K, W + n * K, &y, &mag);\n        if (res)\n            y += oracle_bf16_decode(res[m * N + n]);\n        if (y_ref)",
                         "oracle_point(K, x + m * K, W + n * (K - 1), &y, &mag);\n        if (res)\n            y += oracle_bf16_decode(res[m * N + n]);\n        if (y_ref)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation target for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as d:
        msrc = os.path.join(d, "mutant.c")
        with open(msrc, "w") as f:
            f.write(src.replace(old, new))
        lib = O.load(O.build(msrc, os.path.join(d, f"lib_{name}.so")))
        caught = []
        for check in P.ALL_CHECKS:
            try:
                check(lib)
            except AssertionError:
                caught.append(check.__name__)
        assert caught, f"no pin detects the mutant {name}"
