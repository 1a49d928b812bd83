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
    ("drop_first_term", "for (n = 0; n < N; ++n)\n        s += exp",
     "for (n = 1; n < N; ++n)\n        s += exp"),
    ("drop_last_term", "for (n = 0; n < N; ++n)\n        s += exp",
     "for (n = 0; n + 1 < N; ++n)\n        s += exp"),
    ("wrong_sign_log", "return m + log(s);", "return m - log(s);"),
    ("wrong_sign_shift", "- m);", "+ m);"),
    ("min_not_max", "else if (v > m)", "else if (v < m && v > -INFINITY)"),
    ("missing_nan_rule", "    if (any_nan)\n        return NAN;\n", ""),
    ("missing_pos_inf_rule", "    if (any_pos_inf)\n        return INFINITY;\n", ""),
    ("log2_not_ln", "return m + log(s);", "return m + log2(s);"),
    ("stride_ignored", "base + b * row_stride * es", "base + b * N * es"),
    ("f16_bias", "(int)e - 25", "(int)e - 24"),
    ("f16_subnormal", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    ("bf16_shift", "(uint32_t)h << 16", "(uint32_t)h << 15"),
    ("bf16_as_f16", "case ORACLE_BF16: return decode_bf16", "case ORACLE_BF16: return decode_f16"),
    ("float_accumulator", "double m = -INFINITY, s = 0.0;", "double m = -INFINITY; float s = 0.0f;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
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
