"""Pins for the fp64 oracle: checks against what the mathematics fixes.

Each ``check_*`` takes an oracle object (``.lse(x, dtype, B, N, row_stride)``
and ``.decode(x, dtype)``) and raises AssertionError on a mismatch.  The same
checks run against the real oracle (all must pass) and against deliberately
broken copies of it (at least one must fail), which shows the pins are strong
enough to catch a dropped term, a wrong sign, a wrong index or stride, or a
wrong decode.

Nothing here retypes the oracle's max-subtract-then-sum loop: references are
closed forms, exact invariants, library routines (numpy/torch dtype decodes,
scipy.special.logsumexp) and brute force in 40-digit arithmetic (mpmath).

Source of the definition: "Speeding up Log-Sum-Exp: Kernel Fusion at the
Memory Wall, Integer Arithmetic at the Compute Wall", TL;DR and Sec. 2; the
pairwise operation is associative and commutative (Sec. 3.1).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

try:
    import mpmath
except ImportError:  # pragma: no cover - mpmath ships with sympy here
    mpmath = None

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _same(got: float, want: float, tol_abs: float, tol_rel: float) -> bool:
    if math.isnan(want):
        return math.isnan(got)
    if math.isinf(want):
        return got == want
    return (not math.isnan(got)) and abs(got - want) <= tol_abs + tol_rel * abs(want)


def _row_array(row, dtype):
    vals = np.array([float(v) for v in row], dtype=np.float64)
    if dtype == "f32":
        return vals.astype(np.float32)[None, :]
    if dtype == "f16":
        return vals.astype(np.float16)[None, :]
    if dtype == "bf16":
        f = vals.astype(np.float32)
        assert np.all((f.view(np.uint32) & 0xFFFF) == 0) or np.all(np.isnan(f)), \
            "bf16 fixture values must be exact"
        return (f.view(np.uint32) >> 16).astype(np.uint16)[None, :]
    raise ValueError(dtype)


def _mp_eval(expr: str) -> float:
    if expr in ("inf", "-inf", "nan"):
        return float(expr)
    mpmath.mp.dps = 40
    return float(mpmath.mpf(eval(expr, {"log": mpmath.log, "e": mpmath.e,
                                        "__builtins__": {}})))


def check_golden(orc) -> None:
    """Closed-form fixtures under tests/golden/closed_forms.json."""
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        row = c["row"] if "row" in c else [c["row_repeat"][0]] * c["row_repeat"][1]
        x = _row_array(row, c["dtype"]) if row else np.zeros((1, 0), np.float32)
        if not row and c["dtype"] != "f32":
            x = np.zeros((1, 0), np.uint16)
        got = float(orc.lse(x, c["dtype"])[0])
        want = _mp_eval(c["expected"])
        assert _same(got, want, 1e-13, 1e-15), (c["name"], got, want)


def check_decode_all_patterns(orc) -> None:
    """Every 16-bit pattern decodes as numpy (f16) / torch (bf16) decode it."""
    import torch

    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want16 = bits.view(np.float16).astype(np.float64)
    got16 = orc.decode(bits, "f16")
    nan = np.isnan(want16)
    assert np.array_equal(np.isnan(got16), nan)
    assert np.array_equal(got16[~nan], want16[~nan])

    wantbf = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16) \
        .to(torch.float64).numpy()
    gotbf = orc.decode(bits, "bf16")
    nan = np.isnan(wantbf)
    assert np.array_equal(np.isnan(gotbf), nan)
    assert np.array_equal(gotbf[~nan], wantbf[~nan])

    f = np.array([0.0, -0.0, 1.0, -2.5, 1e-45, 3.4e38, np.inf, -np.inf, np.nan],
                 dtype=np.float32)
    got = orc.decode(f, "f32")
    assert np.array_equal(np.isnan(got), np.isnan(f.astype(np.float64)))
    assert np.array_equal(got[:-1], f[:-1].astype(np.float64))


def check_single_element_rows(orc) -> None:
    """N = 1: log(exp(x)) = x for every 16-bit pattern (one row per pattern)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in ("f16", "bf16"):
        want = orc.decode(bits, dt)
        got = orc.lse(bits.reshape(-1, 1), dt)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), dt
        assert np.array_equal(got[~nan], want[~nan]), dt


def check_constant_rows(orc) -> None:
    """A constant row c of length N gives c + log N."""
    for n in (1, 2, 3, 7, 64, 1000, 4097, 100003):
        for c in (0.0, -3.5, 12.25, 1000.0, -1000.0, 88.5, -104.0):
            x = np.full((1, n), c, dtype=np.float32)
            got = float(orc.lse(x)[0])
            want = c + math.log(n)
            assert abs(got - want) <= 4e-16 * (1 + abs(want)) + 1e-15 * math.log(n), \
                (n, c, got, want)


def check_special_values(orc) -> None:
    """NaN > +inf > all -inf; -inf entries add nothing; N = 0 gives -inf."""
    inf, nan = np.inf, np.nan
    rows = [
        ([nan], "nan"), ([0.0, nan], "nan"), ([nan, 5.0], "nan"), ([inf, nan], "nan"),
        ([-inf, nan, inf], "nan"), ([inf], "inf"), ([-inf, inf], "inf"),
        ([1e30, inf, -1e30], "inf"), ([-inf], "-inf"), ([-inf] * 9, "-inf"),
    ]
    for r, want in rows:
        got = float(orc.lse(np.array([r], dtype=np.float32))[0])
        assert _same(got, float(want), 0, 0), (r, got, want)
    for n in (2, 5, 33):
        for k in range(n):
            x = np.full((1, n), -inf, dtype=np.float32)
            x[0, k] = 0.0
            assert float(orc.lse(x)[0]) == 0.0, (n, k)
            x[0, k] = nan
            assert math.isnan(float(orc.lse(x)[0])), (n, k)
            x[0, k] = inf
            assert float(orc.lse(x)[0]) == inf, (n, k)
    assert float(orc.lse(np.zeros((3, 0), np.float32))[2]) == -inf
    for dt in ("f16", "bf16"):
        pinf = np.uint16(0x7C00 if dt == "f16" else 0x7F80)
        ninf = np.uint16(0xFC00 if dt == "f16" else 0xFF80)
        qnan = np.uint16(0x7E00 if dt == "f16" else 0x7FC0)
        one = np.uint16(0x3C00 if dt == "f16" else 0x3F80)
        x = np.array([[one, pinf], [one, qnan], [ninf, ninf], [ninf, one]], np.uint16)
        got = orc.lse(x, dt)
        assert got[0] == inf and math.isnan(got[1]) and got[2] == -inf, (dt, got)
        assert got[3] == 1.0, (dt, got)


def check_two_element_closed_form(orc) -> None:
    """lse(a, b) = max(a, b) + log1p(exp(-|a - b|)), in 40-digit arithmetic."""
    mpmath.mp.dps = 40
    rng = np.random.default_rng(7)
    ab = np.concatenate([rng.normal(0, 5, (200, 2)), rng.normal(0, 400, (50, 2))])
    ab = ab.astype(np.float32)
    got = orc.lse(ab)
    for (a, b), g in zip(ab.astype(np.float64), got):
        want = float(max(a, b) + mpmath.log1p(mpmath.exp(-abs(mpmath.mpf(a) - b))))
        assert abs(g - want) <= 4e-16 * (1 + abs(want)), (a, b, g, want)


def check_brute_force(orc) -> None:
    """Tiny rows: log(sum exp(x)) directly in 40-digit arithmetic (no max-subtract)."""
    mpmath.mp.dps = 40
    rng = np.random.default_rng(11)
    for n in range(1, 17):
        x = rng.uniform(-30, 30, (8, n)).astype(np.float32)
        if n > 2:
            x[0, n // 2] = -np.inf
        got = orc.lse(x)
        for row, g in zip(x.astype(np.float64), got):
            want = float(mpmath.log(mpmath.fsum(mpmath.exp(mpmath.mpf(v)) for v in row
                                                if v != -np.inf)))
            assert abs(g - want) <= 1e-14 * max(1.0, abs(want)), (n, g, want)


def check_against_scipy(orc) -> None:
    """scipy.special.logsumexp on random rows, three scales and all dtypes."""
    from scipy.special import logsumexp

    rng = np.random.default_rng(3)
    for scale in (1.0, 30.0, 3000.0):
        x = (rng.normal(0, scale, (32, 999)) + rng.uniform(-50, 50, (32, 1))) \
            .astype(np.float32)
        got = orc.lse(x)
        want = logsumexp(x.astype(np.float64), axis=1)
        assert np.allclose(got, want, rtol=1e-14, atol=1e-13), scale
        h = x.astype(np.float16)
        assert np.allclose(orc.lse(h, "f16"), logsumexp(h.astype(np.float64), axis=1),
                           rtol=1e-14, atol=1e-13)
        bf = (x.view(np.uint32) >> 16).astype(np.uint16)
        bfv = (bf.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.allclose(orc.lse(bf, "bf16"), logsumexp(bfv, axis=1),
                           rtol=1e-14, atol=1e-13)


def check_shift_invariance(orc) -> None:
    """lse(x + c) = lse(x) + c, with x on a 2^-6 grid so x + c is exact in f32."""
    rng = np.random.default_rng(5)
    x = (np.round(rng.uniform(-16, 16, (16, 513)) * 64) / 64).astype(np.float32)
    base = orc.lse(x)
    for c in (1000.0, -1000.0, 1e4, -1e4):
        xs = x + np.float32(c)
        assert np.array_equal(xs.astype(np.float64), x.astype(np.float64) + c)
        got = orc.lse(xs)
        assert np.all(np.abs(got - (base + c)) <= 4e-16 * np.abs(base + c) + 1e-13), c


def check_permutation_invariance(orc) -> None:
    """The pairwise operation is commutative: any order of a row gives one value."""
    rng = np.random.default_rng(9)
    x = rng.normal(0, 10, (8, 777)).astype(np.float32)
    x[:, ::50] = -np.inf
    base = orc.lse(x)
    for _ in range(3):
        p = rng.permutation(x.shape[1])
        assert np.allclose(orc.lse(np.ascontiguousarray(x[:, p])), base,
                           rtol=1e-14, atol=0)
    assert np.allclose(orc.lse(np.ascontiguousarray(x[:, ::-1])), base, rtol=1e-14, atol=0)


def check_split_associativity(orc) -> None:
    """lse(x) = lse2(lse(x[:k]), lse(x[k:])) for every split point k (Sec. 3.1)."""
    mpmath.mp.dps = 40
    rng = np.random.default_rng(13)
    x = rng.normal(0, 6, (1, 97)).astype(np.float32)
    x[0, 40] = 20.0
    whole = float(orc.lse(x)[0])
    for k in range(0, 98):
        a = float(orc.lse(np.ascontiguousarray(x[:, :k]))[0])
        b = float(orc.lse(np.ascontiguousarray(x[:, k:]))[0])
        if a == -np.inf:
            comb = b
        elif b == -np.inf:
            comb = a
        else:
            comb = float(max(a, b) + mpmath.log1p(mpmath.exp(-abs(mpmath.mpf(a) - b))))
        assert abs(comb - whole) <= 1e-14 * abs(whole) + 1e-14, (k, comb, whole)


def check_bounds(orc) -> None:
    """max x <= lse(x) <= max x + log N."""
    rng = np.random.default_rng(17)
    for n in (1, 2, 10, 1000):
        x = rng.normal(0, 20, (50, n)).astype(np.float32)
        got = orc.lse(x)
        m = x.max(axis=1).astype(np.float64)
        assert np.all(got >= m) and np.all(got <= m + math.log(n) + 1e-12), n


def check_row_stride(orc) -> None:
    """Only the first N columns of each padded row are read."""
    rng = np.random.default_rng(19)
    x = rng.normal(0, 3, (9, 100)).astype(np.float32)
    padded = np.full((9, 131), np.nan, dtype=np.float32)
    padded[:, :100] = x
    assert np.array_equal(orc.lse(padded, "f32", 9, 100, 131), orc.lse(x))
    flat = padded.reshape(-1)[: 8 * 131 + 100]
    assert np.array_equal(orc.lse(flat, "f32", 9, 100, 131), orc.lse(x))


# ---------------------------------------------------------------------------
# Token log-probability: logprob[b] = x[b, t] - lse[b]
# ---------------------------------------------------------------------------
def check_logprob_closed_forms(orc) -> None:
    """Constant row: -log N; one-hot: 0 at the hot column, -inf elsewhere;
    targets outside [0, N): NaN; a NaN row: NaN."""
    for n in (1, 3, 1000):
        for c in (0.0, -7.25, 1000.0):
            x = np.full((n, n), c, dtype=np.float32)
            lp, lse = orc.token_logprob(x, np.arange(n))
            assert np.all(np.abs(lp + math.log(n)) <= 1e-15 * (1 + abs(c))), (n, c)
    x = np.full((4, 6), -np.inf, dtype=np.float32)
    x[:, 2] = 0.0
    lp, _ = orc.token_logprob(x, np.array([2, 0, 5, 2]))
    assert lp[0] == 0.0 and lp[3] == 0.0 and lp[1] == -np.inf and lp[2] == -np.inf, lp
    y = np.zeros((5, 4), dtype=np.float32)
    lp, _ = orc.token_logprob(y, np.array([-1, 4, 1 << 40, -(1 << 40), 3]))
    assert np.all(np.isnan(lp[:4])) and abs(lp[4] + math.log(4)) < 1e-15, lp
    y[1, 0] = np.nan
    lp, _ = orc.token_logprob(y[:2], np.array([1, 1]))
    assert not math.isnan(lp[0]) and math.isnan(lp[1])


def check_logprob_normalizes(orc) -> None:
    """sum over every target t of exp(logprob_t) = 1 (40-digit sum)."""
    mpmath.mp.dps = 40
    rng = np.random.default_rng(23)
    for n in (2, 17, 300):
        row = rng.normal(0, 8, n).astype(np.float32)
        lp, _ = orc.token_logprob(np.tile(row, (n, 1)), np.arange(n))
        total = mpmath.fsum(mpmath.exp(mpmath.mpf(v)) for v in lp)
        assert abs(float(total) - 1.0) <= 1e-13, (n, float(total))


def check_logprob_against_scipy(orc) -> None:
    from scipy.special import logsumexp

    rng = np.random.default_rng(29)
    x = (rng.normal(0, 5, (64, 777)) + rng.uniform(-30, 30, (64, 1))).astype(np.float32)
    t = rng.integers(0, 777, 64)
    lp, lse = orc.token_logprob(x, t)
    want_lse = logsumexp(x.astype(np.float64), axis=1)
    want = x[np.arange(64), t].astype(np.float64) - want_lse
    assert np.allclose(lse, want_lse, rtol=1e-14, atol=1e-13)
    assert np.allclose(lp, want, rtol=1e-12, atol=1e-12)


def check_logprob_shift_invariance(orc) -> None:
    rng = np.random.default_rng(31)
    x = (np.round(rng.uniform(-16, 16, (8, 129)) * 64) / 64).astype(np.float32)
    t = rng.integers(0, 129, 8)
    base, _ = orc.token_logprob(x, t)
    for c in (1000.0, -1000.0):
        got, _ = orc.token_logprob(x + np.float32(c), t)
        assert np.all(np.abs(got - base) <= 1e-12), c


# ---------------------------------------------------------------------------
# Backward: dx[b, n] = g[b] * exp(x[b, n] - lse[b])
# ---------------------------------------------------------------------------
def check_backward_sums_to_grad(orc) -> None:
    """Each row of exp(x - lse) is a probability vector: sum_n dx[b, n] = g[b]."""
    rng = np.random.default_rng(37)
    x = rng.normal(0, 6, (16, 513)).astype(np.float32)
    x[3, ::7] = -np.inf
    g = rng.normal(0, 2, 16)
    dx = orc.backward(x, orc.lse(x), g)
    assert np.allclose(dx.sum(axis=1), g, rtol=1e-13, atol=1e-13)
    assert np.all(dx[3, ::7] == 0.0)


def check_backward_finite_difference(orc) -> None:
    """d lse / d x[n] by central differences of the forward oracle (x on a 2^-10
    grid, step 2^-10, both exact in f32) matches exp(x[n] - lse)."""
    rng = np.random.default_rng(41)
    x = (np.round(rng.uniform(-4, 4, (3, 9)) * 1024) / 1024).astype(np.float32)
    h = 2.0 ** -10
    dx = orc.backward(x, orc.lse(x), np.ones(3))
    for b in range(3):
        for n in range(9):
            xp, xm = x[b:b + 1].copy(), x[b:b + 1].copy()
            xp[0, n] += np.float32(h)
            xm[0, n] -= np.float32(h)
            fd = (orc.lse(xp)[0] - orc.lse(xm)[0]) / (2 * h)
            assert abs(fd - dx[b, n]) <= 2e-7, (b, n, fd, dx[b, n])


def check_backward_against_scipy(orc) -> None:
    from scipy.special import softmax

    rng = np.random.default_rng(43)
    x = (rng.normal(0, 4, (32, 200)) + rng.uniform(-50, 50, (32, 1))).astype(np.float32)
    g = rng.normal(0, 1, 32)
    for dt in ("f32", "bf16", "f16"):
        if dt == "f32":
            xx, xv = x, x.astype(np.float64)
        elif dt == "f16":
            xx = x.astype(np.float16)
            xv = xx.astype(np.float64)
        else:
            xx = (x.view(np.uint32) >> 16).astype(np.uint16)
            xv = (xx.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        dx = orc.backward(xx, orc.lse(xx, dt), g, dt)
        assert np.allclose(dx, g[:, None] * softmax(xv, axis=1), rtol=1e-12, atol=1e-15), dt


def check_backward_special(orc) -> None:
    """One-hot rows give g at the hot column; an all -inf row gives NaN
    (exp(-inf - (-inf))), as the plain formula does in IEEE arithmetic."""
    x = np.full((2, 5), -np.inf, dtype=np.float32)
    x[0, 3] = 2.0
    dx = orc.backward(x, orc.lse(x), np.array([1.5, 1.0]))
    assert np.array_equal(dx[0], [0, 0, 0, 1.5, 0]) and np.all(np.isnan(dx[1]))


# ---------------------------------------------------------------------------
# Strided: out[a, c] = log sum_r exp(x[a*sa + r*sr + c])
# ---------------------------------------------------------------------------
def check_strided_against_scipy(orc) -> None:
    """LSE over dim 1 of an [A, R, C] array, contiguous and padded, all dtypes."""
    from scipy.special import logsumexp

    rng = np.random.default_rng(47)
    A, R, C = 3, 37, 21
    x = (rng.normal(0, 6, (A, R, C)) + rng.uniform(-40, 40, (A, 1, C))).astype(np.float32)
    want = logsumexp(x.astype(np.float64), axis=1)
    got = orc.lse_strided(x.reshape(-1), "f32", A, R, C, R * C, C)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-13)
    pad = np.full((A, R + 2, C + 5), np.nan, np.float32)  # padded strides: never read
    pad[:, :R, :C] = x
    got = orc.lse_strided(pad.reshape(-1), "f32", A, R, C, (R + 2) * (C + 5), C + 5)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-13)
    h = x.astype(np.float16)
    got = orc.lse_strided(h.reshape(-1), "f16", A, R, C, R * C, C)
    assert np.allclose(got, logsumexp(h.astype(np.float64), axis=1), rtol=1e-14, atol=1e-13)


def check_strided_matches_rows(orc) -> None:
    """A column of a matrix is the row of its transpose; stride_r = 1 with C = 1
    is a row; R = 0 gives -inf; special values per column."""
    rng = np.random.default_rng(53)
    m = rng.normal(0, 4, (50, 9)).astype(np.float32)
    m[:, 2] = -np.inf
    m[7, 3] = np.nan
    m[9, 4] = np.inf
    m[:, 5] = -np.inf
    m[11, 5] = 1.5
    cols = orc.lse_strided(m.reshape(-1), "f32", 1, 50, 9, 0, 9)[0]
    rows = orc.lse(np.ascontiguousarray(m.T))
    assert np.array_equal(np.isnan(cols), np.isnan(rows))
    assert np.array_equal(cols[~np.isnan(cols)], rows[~np.isnan(rows)])
    assert cols[2] == -np.inf and np.isnan(cols[3]) and cols[4] == np.inf and cols[5] == 1.5
    r = rng.normal(0, 4, 30).astype(np.float32)
    assert orc.lse_strided(r, "f32", 1, 30, 1, 0, 1)[0, 0] == orc.lse(r[None, :])[0]
    assert np.all(orc.lse_strided(r, "f32", 2, 0, 3, 0, 0) == -np.inf)


def check_strided_backward_sums_to_grad(orc) -> None:
    """Over the reduced dimension exp(x - lse) sums to 1: sum_r dx[a, r, c] = g[a, c];
    -inf entries get 0."""
    rng = np.random.default_rng(59)
    A, R, C = 3, 41, 17
    x = (rng.normal(0, 5, (A, R, C)) + rng.uniform(-30, 30, (A, 1, C))).astype(np.float32)
    x[1, ::5, 4] = -np.inf
    lse = orc.lse_strided(x.reshape(-1), "f32", A, R, C, R * C, C)
    g = rng.normal(0, 2, (A, C))
    dx = orc.backward_strided(x.reshape(-1), "f32", A, R, C, R * C, C, lse, g)
    assert np.allclose(dx.sum(axis=1), g, rtol=1e-13, atol=1e-13)
    assert np.all(dx[1, ::5, 4] == 0.0)


def check_strided_backward_finite_difference(orc) -> None:
    """d out[a, c] / d x[a, r, c] by central differences of the strided forward
    oracle (x on a 2^-10 grid, step 2^-10, exact in f32), on a padded layout;
    other columns do not move."""
    rng = np.random.default_rng(61)
    A, R, C = 2, 5, 3
    sa, sr = R * (C + 2) + 3, C + 2
    x = (np.round(rng.uniform(-4, 4, (A, R, C)) * 1024) / 1024).astype(np.float32)
    buf = np.full((A - 1) * sa + (R - 1) * sr + C + 4, np.nan, np.float32)
    for a in range(A):
        for r in range(R):
            buf[a * sa + r * sr:a * sa + r * sr + C] = x[a, r]
    lse = orc.lse_strided(buf, "f32", A, R, C, sa, sr)
    dx = orc.backward_strided(buf, "f32", A, R, C, sa, sr, lse, np.ones((A, C)))
    h = 2.0 ** -10
    for a in range(A):
        for r in range(R):
            for c in range(C):
                bp, bm = buf.copy(), buf.copy()
                bp[a * sa + r * sr + c] += np.float32(h)
                bm[a * sa + r * sr + c] -= np.float32(h)
                lp = orc.lse_strided(bp, "f32", A, R, C, sa, sr)
                lm = orc.lse_strided(bm, "f32", A, R, C, sa, sr)
                fd = (lp - lm) / (2 * h)
                assert abs(fd[a, c] - dx[a, r, c]) <= 2e-7, (a, r, c)
                others = np.ones((A, C), bool)
                others[a, c] = False
                assert np.all(fd[others] == 0.0)


def check_strided_backward_matches_rows(orc) -> None:
    """A column's gradient is the row gradient of the transpose, special values
    included; bf16 and f16 decode as in the row oracle."""
    rng = np.random.default_rng(67)
    m = rng.normal(0, 4, (30, 7)).astype(np.float32)
    m[:, 2] = -np.inf
    m[4, 3] = np.nan
    m[6, 5] = np.inf
    g = rng.normal(0, 1, 7)
    lse = orc.lse_strided(m.reshape(-1), "f32", 1, 30, 7, 0, 7)
    cols = orc.backward_strided(m.reshape(-1), "f32", 1, 30, 7, 0, 7, lse, g[None, :])[0]
    rows = orc.backward(np.ascontiguousarray(m.T), lse[0], g)
    assert np.array_equal(np.isnan(cols), np.isnan(rows.T))
    ok = ~np.isnan(cols)
    assert np.array_equal(cols[ok], rows.T[ok])
    for dt in ("f16", "bf16"):
        h = m.astype(np.float16) if dt == "f16" else (m.view(np.uint32) >> 16).astype(np.uint16)
        lh = orc.lse_strided(h.reshape(-1), dt, 1, 30, 7, 0, 7)
        ch = orc.backward_strided(h.reshape(-1), dt, 1, 30, 7, 0, 7, lh, g[None, :])[0]
        rh = orc.backward(np.ascontiguousarray(h.T), lh[0], g, dt)
        ok = ~np.isnan(ch)
        assert np.array_equal(np.isnan(ch), np.isnan(rh.T)) and np.array_equal(ch[ok], rh.T[ok])


ALL_CHECKS = [
    check_golden, check_decode_all_patterns, check_single_element_rows,
    check_constant_rows, check_special_values, check_two_element_closed_form,
    check_brute_force, check_against_scipy, check_shift_invariance,
    check_permutation_invariance, check_split_associativity, check_bounds,
    check_row_stride, check_logprob_closed_forms, check_logprob_normalizes,
    check_logprob_against_scipy, check_logprob_shift_invariance,
    check_backward_sums_to_grad, check_backward_finite_difference,
    check_backward_against_scipy, check_backward_special,
    check_strided_against_scipy, check_strided_matches_rows,
    check_strided_backward_sums_to_grad, check_strided_backward_finite_difference,
    check_strided_backward_matches_rows,
]
