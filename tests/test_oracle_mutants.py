"""Planted mistakes in copies of the oracle must fail at least one pin.

Each mutant is the oracle's C source with one plausible error patched in (a
dropped term, a wrong sign, a wrong index or stride, a broken decode, a missed
special value), compiled with gcc on the CPU.  The real oracle is never
changed.  A mutant that passes every pin would show a hole in the pins.
"""
import os
import subprocess

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "lse_oracle.c")

# (name, text in the oracle, replacement)
MUTANTS = [
    ("drop_first_term", "for (n = 0; n < count; ++n)\n        s += exp",
     "for (n = 1; n < count; ++n)\n        s += exp"),
    ("wrong_sign_log", "return m + log(s);", "return m - log(s);"),
    ("wrong_sign_shift", "n * step) - m);", "n * step) + m);"),
    ("min_not_max", "else if (v > m)", "else if (v < m && v > -INFINITY)"),
    ("row_step_two", "return lse_strided(dtype, row, N, 1);", "return lse_strided(dtype, row, N / 2, 2);"),
    ("missing_nan_rule", "    if (any_nan)\n        return NAN;\n", ""),
    ("missing_pos_inf_rule", "    if (any_pos_inf)\n        return INFINITY;\n", ""),
    ("log2_not_ln", "return m + log(s);", "return m + log2(s);"),
    ("stride_ignored", "lse_row(dtype, base + b * row_stride * es, N)",
     "lse_row(dtype, base + b * N * es, N)"),
    ("f16_bias", "(int)e - 25", "(int)e - 24"),
    ("f16_subnormal", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    ("bf16_shift", "(uint32_t)h << 16", "(uint32_t)h << 15"),
    ("bf16_as_f16", "case ORACLE_BF16: return decode_bf16", "case ORACLE_BF16: return decode_f16"),
    ("float_accumulator", "double m = -INFINITY, s = 0.0;", "double m = -INFINITY; float s = 0.0f;"),
    ("logprob_sign", "decode(dtype, row, t) - v : NAN", "v - decode(dtype, row, t) : NAN"),
    ("logprob_drops_target_0", "(t >= 0 && t < N)", "(t > 0 && t < N)"),
    ("logprob_wrong_column", "decode(dtype, row, t) - v", "decode(dtype, row, t > 0 ? t - 1 : t) - v"),
    ("logprob_first_row_lse", "const double v = lse_row(dtype, row, N);",
     "const double v = lse_row(dtype, base, N);"),
    ("backward_no_grad", "= grad[b] * exp(decode", "= exp(decode"),
    ("backward_sign", "exp(decode(dtype, row, n) - lse[b])", "exp(lse[b] - decode(dtype, row, n))"),
    ("backward_first_row_lse", "n) - lse[b])", "n) - lse[0])"),
    ("strided_ignores_step", "decode(dtype, base, n * step);", "decode(dtype, base, n);"),
    ("strided_swaps_a_and_c", "base + (a * stride_a + c) * es", "base + (c * stride_a + a) * es"),
    ("strided_drops_last", "for (n = 0; n < count; ++n)\n        s += exp",
     "for (n = 0; n + 1 < count; ++n)\n        s += exp"),
    ("strided_backward_row_lse", "- lse[a * C + c]);", "- lse[a * C]);"),
    ("strided_backward_ignores_step", "base + (a * stride_a + r * stride_r) * es",
     "base + (a * stride_a + r * C) * es"),
    ("strided_backward_no_grad", "grad[a * C + c] * exp(", "exp("),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} must occur exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(mutated), "-lm"], check=True)
    mutant = oracle.OracleLib(str(so))
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(mutant)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
