"""Helpers shared by the GPU tests: tolerance check and device layouts."""
from __future__ import annotations

import numpy as np

# Parity bar for finite outputs: |gpu - oracle| <= ATOL + RTOL * |oracle|;
# NaN and +-inf must match exactly.
ATOL = 1e-5
RTOL = 1e-6


def compare(got: np.ndarray, want: np.ndarray, atol: float = ATOL, rtol: float = RTOL,
            scale: np.ndarray | None = None) -> dict:
    """Compare float32 GPU results with float64 oracle values; return a summary.

    Finite values must satisfy |got - want| <= atol + rtol * scale, where scale
    defaults to |want|.
    """
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    nan_w, nan_g = np.isnan(want), np.isnan(got)
    bad_nan = np.flatnonzero(nan_w != nan_g)
    inf_w = np.isinf(want)
    bad_inf = np.flatnonzero(inf_w & ~nan_g & (got != want))
    fin = ~nan_w & ~inf_w
    err = np.abs(got[fin] - want[fin])
    sc = np.abs(want) if scale is None else np.abs(np.asarray(scale, dtype=np.float64))
    lim = atol + rtol * sc[fin]
    bad_fin = np.flatnonzero(fin)[~(err <= lim)]
    summary = {
        "n": int(got.size),
        "finite": int(fin.sum()),
        "max_abs_err": float(err.max()) if err.size else 0.0,
        "max_err_over_tol": float((err / lim).max()) if err.size and lim.min() > 0 else 0.0,
    }
    if bad_nan.size or bad_inf.size or bad_fin.size:
        idx = np.concatenate([bad_nan, bad_inf, bad_fin])[:8]
        detail = [(int(i), float(got.flat[i]), float(want.flat[i])) for i in idx]
        raise AssertionError(f"{bad_nan.size} NaN mismatches, {bad_inf.size} inf mismatches, "
                             f"{bad_fin.size} out of tolerance; first: {detail}; {summary}")
    return summary


def torch_view(x: np.ndarray, dtype: str):
    """A torch CPU tensor with the raw bits of ``x`` in the matching dtype."""
    import torch

    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    if dtype == "f16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.float16)
    raise ValueError(dtype)


def compare_logprob(got_lp: np.ndarray, want_lp: np.ndarray, want_lse: np.ndarray) -> dict:
    """Token log-probabilities: the row value's error carries over, so the bar
    is |d| <= ATOL + RTOL * (|logprob| + |lse|) (>= the bar on x[b, t] - lse)."""
    scale = np.abs(np.nan_to_num(want_lp, posinf=0, neginf=0)) + \
        np.abs(np.nan_to_num(want_lse, posinf=0, neginf=0))
    return compare(got_lp, want_lp, ATOL, RTOL, scale)


NAN_BITS = {"f32": None, "bf16": 0x7FC0, "f16": 0x7E00}


def canary_array(shape, dtype: str) -> np.ndarray:
    """A host array of NaNs (raw bits for 16-bit types)."""
    if dtype == "f32":
        return np.full(shape, np.nan, dtype=np.float32)
    return np.full(shape, NAN_BITS[dtype], dtype=np.uint16)


def device_rows(x: np.ndarray, dtype: str, row_stride: int | None = None, offset: int = 0,
                device: str = "cuda"):
    """Place [B, N] rows on the device inside a NaN-filled buffer.

    Rows start ``offset`` elements into the buffer, ``row_stride`` apart; every
    element outside the rows (padding, before, after) is NaN, so a kernel that
    reads outside [0, N) of a row returns NaN for it.  Returns (buffer, view).
    """
    import torch

    B, N = x.shape
    row_stride = N if row_stride is None else row_stride
    total = offset + B * row_stride + 64
    host = canary_array(total, dtype)
    if B:
        body = host[offset:offset + B * row_stride].reshape(B, row_stride)
        body[:, :N] = x if dtype == "f32" else np.ascontiguousarray(x).view(np.uint16)
    buf = torch_view(host, dtype).to(device)
    if B == 0:
        return buf, buf[offset:offset].reshape(0, N)
    view = buf[offset:offset + B * row_stride].reshape(B, row_stride)[:, :N]
    return buf, view


# Reduced-bit exponentials (lse_forward16): a term with base-2 argument a is
# within a relative r(a) = 2^(E16_BIAS + (|a| + E16_BIAS) E16_ARG) - 1 + E16_OUT
# of its exact value (the accuracy statement of lse_forward16 in include/lse.h):
# the argument carries the constant E16_BIAS and is rounded to bf16, and the
# SFU's bf16 result is truncated (by less than a factor 1 - E16_OUT).
E16_ARG = 2.0 ** -8 + 2.0 ** -22  # bf16 rounding of the argument, plus its f32 steps
E16_OUT = 2.0 ** -7               # truncation of the packed bf16 exponential's result
E16_BIAS = 0.0040709119223702435  # -log2(1 - 2^-8 / (2 ln 2))
LOG2E = 1.4426950408889634


def e16_bound(x: np.ndarray, dtype: str, want: np.ndarray, block_elems: int = 1 << 24):
    """Per-row bound on |lse_forward16 - oracle|: -log(1 - e) + ATOL + RTOL |want|
    with e = e16_error_sum(...).  inf for non-finite rows (those must match
    exactly)."""
    e = e16_error_sum(x, dtype, want, block_elems)
    want = np.asarray(want, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        bnd = np.where(e < 1.0, -np.log1p(-np.minimum(e, 0.999999)), np.inf)
    return np.where(np.isfinite(want), bnd + ATOL + RTOL * np.abs(want), np.inf)


def e16_error_sum(x: np.ndarray, dtype: str, want: np.ndarray, block_elems: int = 1 << 24,
                  row_max: np.ndarray | None = None):
    """e = sum_n p_n r(a_n) per row: p the oracle's softmax of the row (its
    backward with unit gradient, against the row value ``want``) and
    |a_n| = (max - x_n) log2 e.  ``row_max`` overrides the maximum (for a
    slice of a longer row).  nan for non-finite rows."""
    import oracle

    B = want.shape[0]
    N = x.shape[1] if x.ndim == 2 else 0
    out = np.full(B, np.nan)
    rows = max(1, block_elems // max(N, 1))
    for b0 in range(0, B, rows):
        xb = np.ascontiguousarray(x[b0:b0 + rows])
        wb = np.asarray(want[b0:b0 + rows], dtype=np.float64)
        fin = np.isfinite(wb)
        if not fin.any() or N == 0:
            continue
        xd = oracle.decode(xb, dtype).reshape(xb.shape[0], N)
        p = oracle.backward(xb, np.where(fin, wb, 0.0), np.ones(len(wb)), dtype)
        p = p.reshape(xb.shape[0], N)
        m = np.max(np.where(np.isnan(xd), -np.inf, xd), axis=1) if row_max is None \
            else np.asarray(row_max, dtype=np.float64)[b0:b0 + len(wb)]
        with np.errstate(invalid="ignore", over="ignore"):
            a = (m[:, None] - xd) * LOG2E
            r = np.exp2(E16_BIAS + (a + E16_BIAS) * E16_ARG) - 1.0 + E16_OUT
            r = np.where(a > 125.0, 1.0, r)  # flushed below 2^-126 of the maximum
            e = np.where(p > 0, p * r, 0.0).sum(axis=1)
        out[b0:b0 + len(wb)] = np.where(fin, e, np.nan)
    return out


def compare_e16(got: np.ndarray, want: np.ndarray, bound: np.ndarray) -> dict:
    """Special values exactly, finite rows within their e16_bound; the summary
    adds the mean absolute and mean signed errors."""
    s = compare(got, want, atol=0.0, rtol=1.0, scale=bound)
    fin = np.isfinite(np.asarray(want, dtype=np.float64))
    d = np.asarray(got, dtype=np.float64)[fin] - np.asarray(want, dtype=np.float64)[fin]
    s["mean_abs_err"] = float(np.abs(d).mean()) if d.size else 0.0
    s["mean_err"] = float(d.mean()) if d.size else 0.0
    return s


# Backward: dx = g exp(x - lse) computed in f32 and rounded once to the element
# type.  Relative bar per element: the f32 steps (2^-21 plus 2^-23 per unit of
# |lse| and |x - lse|, the argument's rounding) plus the output rounding q, an
# absolute 1e-37 |g| for flushed results and 2^-24 for f16 subnormals.
BWD_Q = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def compare_backward(got: np.ndarray, xv: np.ndarray, dtype: str, lse64: np.ndarray,
                     g: np.ndarray, want: np.ndarray) -> float:
    """got, xv: decoded float64 [B, n] dx and x; want: the oracle's dx.  Special
    values exactly; returns the largest error / bar."""
    nan_w, nan_g = np.isnan(want), np.isnan(got)
    assert np.array_equal(nan_w, nan_g), f"NaN mismatch at {np.argwhere(nan_w != nan_g)[:5]}"
    inf_w = np.isinf(want)
    assert np.array_equal(got[inf_w], want[inf_w])
    fin = ~nan_w & ~inf_w
    lse_b = np.broadcast_to(np.abs(np.nan_to_num(lse64, posinf=0, neginf=0))[:, None], want.shape)
    dist = np.abs(np.nan_to_num(xv - lse64[:, None], posinf=0, neginf=0))
    rel = 2.0 ** -21 + 2.0 ** -23 * (lse_b + dist) + BWD_Q[dtype]
    lim = np.abs(g)[:, None] * 1e-37 + np.abs(want) * rel + (2.0 ** -24 if dtype == "f16" else 0)
    err = np.abs(got - want)
    bad = fin & ~(err <= lim)
    assert not bad.any(), (f"{bad.sum()} out of tolerance; first "
                           f"{[(tuple(i), got[tuple(i)], want[tuple(i)]) for i in np.argwhere(bad)[:4]]}")
    return float((err[fin] / np.maximum(lim[fin], 1e-300)).max()) if fin.any() else 0.0
