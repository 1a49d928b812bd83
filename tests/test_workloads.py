"""Statistical sanity of the seeded workload generators (CPU only).

Not parity: these catch generator mistakes (wrong scale, shift, spike, or
special-value pattern) by comparing the oracle's row values with what each
recipe implies, and check that the draws are deterministic.
"""
import math

import numpy as np

import oracle
from log_sum_exp_gb300 import workloads as wl


def test_deterministic():
    a = wl.generate("small_64x4096_f32")
    b = wl.generate("small_64x4096_f32")
    assert a.dtype == np.float32 and a.shape == (64, 4096)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, wl.generate("small_64x4096_f32", seed=1))


def test_small_normal_rows():
    # E[exp(z)] = e^{1/2} for z ~ N(0,1): lse ~ log N + 1/2.
    got = oracle.lse(wl.generate("small_64x4096_f32"))
    assert abs(got.mean() - (math.log(4096) + 0.5)) < 0.02


def test_vocab128k_spike_rows():
    x = wl.generate("vocab_512x128256_f32", B=8)
    m = x.max(axis=1).astype(np.float64)
    got = oracle.lse(x)
    # spike o+15 is the row max; lse - max = log(1 + N e^{4.5} / e^{15}).
    # e^{3z} is heavy-tailed (sd of the row sum ~20% of its mean at this N).
    want = math.log(1 + 128256 * math.exp(4.5 - 15))
    assert np.all(np.abs((got - m) - want) < 0.25)
    assert abs(np.mean(got - m) - want) < 0.1


def test_vocab32k_bf16_shifted_quarters():
    x = wl.generate("vocab_8192x32000_bf16", B=16, N=32000)
    assert x.dtype == np.uint16
    got = oracle.lse(x, "bf16")
    base = math.log(32000) + 2.0  # E[exp(2z)] = e^2
    # Near |x| = 1000 bf16 values sit on a grid of 4, which raises E[exp(x)]:
    # E = sum_k e^{4k - c} P(c + 2z rounds to 4k), c = +-1000.
    from scipy.stats import norm
    k = np.arange(-15, 16)
    p = norm.cdf((4 * k + 2) / 2.0) - norm.cdf((4 * k - 2) / 2.0)
    quant = math.log(32000 * float(np.sum(np.exp(4.0 * k) * p)))
    assert np.all(np.abs(got[:4] - (1000 + quant)) < 0.15)
    assert np.all(np.abs(got[4:8] - (-1000 + quant)) < 0.15)
    assert np.all(np.abs(got[8:] - base) < 0.1)


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.00390625, 1.01171875, 1.0 + 2 ** -8 + 2 ** -20, -3.0], np.float32)
    bits = wl.f32_to_bf16_bits(f)
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC040]


def test_short_rows_special_pattern():
    B = 200000
    x = wl.generate("short_1048576x32_f32", B=B)
    all_ninf = np.all(x == -np.inf, axis=1)
    has_nan = np.any(np.isnan(x), axis=1)
    assert all_ninf.sum() >= B // 1000 and has_nan.sum() == B // 100000
    assert not np.any(all_ninf & has_nan)
    finite = x[np.isfinite(x)]
    assert finite.min() >= -30 and finite.max() <= 0
    frac = np.mean(x[~all_ninf] == -np.inf)
    assert abs(frac - 0.1) < 0.005
    got = oracle.lse(x)
    assert np.array_equal(np.isnan(got), has_nan)
    assert np.array_equal(got == -np.inf, all_ninf)


def test_particles_rows():
    N = 1 << 20
    x = wl.generate("particles_16x16777216_f32", B=4, N=N)
    assert np.all(x.max(axis=1) == 0.0)
    got = oracle.lse(x)
    want = math.log(1 + (N - 1) / 50 * (1 - math.exp(-50)))
    assert np.all(np.abs(got - want) < 0.02)


def test_random_rows_dtypes():
    for dt, npdt in (("f32", np.float32), ("bf16", np.uint16), ("f16", np.float16)):
        x = wl.random_rows(3, 10, dt, seed=1)
        assert x.dtype == npdt and x.shape == (3, 10)
