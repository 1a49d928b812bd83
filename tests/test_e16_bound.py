"""The per-row error bound used for lse_forward16 (e16_bound), checked on the
CPU against an emulation of its arithmetic: arguments (x - max) log2 e + d in
f32, rounded to bf16; terms 2^a truncated to bf16; sums exact.  A bound that
misses the argument rounding, the constant d, the truncation or the softmax
weighting fails here."""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import E16_BIAS, LOG2E, e16_bound


def _bf16_round(v: np.ndarray) -> np.ndarray:
    """Nearest-even bf16 of float32 values (finite or inf), as float64."""
    bits = wl.f32_to_bf16_bits(v.astype(np.float32)).astype(np.uint32) << np.uint32(16)
    return bits.view(np.float32).astype(np.float64)


def _bf16_trunc(t: np.ndarray) -> np.ndarray:
    """Positive float64 values truncated to 8 significant bits (bf16 toward zero)."""
    m, e = np.frexp(t)
    return np.ldexp(np.floor(m * 256.0) / 256.0, e)


def _emulate(x: np.ndarray) -> np.ndarray:
    """m + log(sum trunc_bf16(2^bf16(fl32((x - m) log2 e + d)))) per row, in float64."""
    m = x.max(axis=1).astype(np.float32)
    d = (x - m[:, None]).astype(np.float32).astype(np.float64)
    a = (d * float(np.float32(LOG2E)) + float(np.float32(E16_BIAS))).astype(np.float32)
    t = _bf16_trunc(np.exp2(_bf16_round(a)))
    return m.astype(np.float64) + np.log(t.sum(axis=1))


@pytest.mark.parametrize("B,N,scale,shift", [(64, 4096, 1.0, 0.0), (16, 128256, 3.0, -20.0),
                                             (256, 32, 10.0, 5.0), (8, 20000, 30.0, 100.0)])
def test_bound_covers_emulated_rounding(B, N, scale, shift):
    x = wl.random_rows(B, N, "f32", seed=N, scale=scale, shift=shift)
    want = oracle.lse(x, "f32")
    bound = e16_bound(x, "f32", want)
    err = np.abs(_emulate(x) - want)
    assert np.all(err <= bound), (err.max(), bound[np.argmax(err / bound)])
    # not vacuous: first order it is at most 2^-7 + 2^-8 ln N (+ f32 terms)
    assert np.all(bound <= 2.0 ** -7 + 2.0 ** -8 * np.log(N) + 1e-3)


def _one_sided_row(a: float, N: int) -> np.ndarray:
    """A row: 0 once, then N - 1 elements whose base-2 argument is a."""
    x = np.full((1, N), np.float32(a / LOG2E), dtype=np.float32)
    x[0, 0] = 0.0
    return x


def test_one_sided_argument_rounding():
    """Every argument plus d is 8 (1 + 0.98 2^-8), which bf16 rounds to 8 by
    almost the largest relative step it allows (2^-8), and 2^-8 truncates
    exactly: the row value moves by ~2.4%, and the bound holds with little room
    (a bound with half the argument term, or without d or the softmax weight,
    fails here)."""
    N = 1 << 16
    x = _one_sided_row(-8.0 * (1.0 + 0.98 * 2.0 ** -8) - E16_BIAS, N)
    want = oracle.lse(x, "f32")
    err = np.abs(_emulate(x) - want)[0]
    bound = e16_bound(x, "f32", want)[0]
    assert 0.6 * bound <= err <= bound, (err, bound)


def test_one_sided_result_rounding():
    """Arguments whose 2^a' truncates by nearly the most bf16 allows: the
    bound still holds, and without the truncation term it would not."""
    grid = -np.arange(1, 256, dtype=np.float64) / 256.0  # bf16 values in (-1, 0)
    t = np.exp2(grid)
    rel = 1.0 - _bf16_trunc(t) / t
    a = float(grid[np.argmax(rel)])
    assert rel.max() > 2.0 ** -8
    x = _one_sided_row(a - E16_BIAS, 4096)
    want = oracle.lse(x, "f32")
    err = np.abs(_emulate(x) - want)[0]
    assert err <= e16_bound(x, "f32", want)[0]


def test_bias_constant_centres_truncation():
    """d makes truncated terms unbiased on average over arguments spread
    evenly, and leaves the maximum's own term exactly 1."""
    rng = np.random.default_rng(7)
    a = -rng.uniform(0.0, 1.0, 200000)
    x = (a / LOG2E).astype(np.float32)[None, :]
    x = np.concatenate([np.zeros((1, 1), np.float32), x], axis=1)
    m = np.float32(0.0)
    d = (x - m).astype(np.float32).astype(np.float64)
    arg = (d * float(np.float32(LOG2E)) + float(np.float32(E16_BIAS))).astype(np.float32)
    t = _bf16_trunc(np.exp2(_bf16_round(arg)))
    exact = np.exp2(d * LOG2E)
    assert t[0, 0] == 1.0
    assert abs(np.mean(t / exact) - 1.0) < 3e-4
    # without d the same terms are 2^-8 / (2 ln 2) = 0.28 % low on average
    t0 = _bf16_trunc(np.exp2(_bf16_round((d * float(np.float32(LOG2E))).astype(np.float32))))
    assert np.mean(t0 / exact) - 1.0 < -2e-3
