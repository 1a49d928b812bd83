"""Reduced-bit exponentials (lse_forward16, the 16-bit compute variant of
"Speeding up Log-Sum-Exp ...", Sec. 4.3 / Fig. 5) against the fp64 oracle.

The value is the plain log-sum-exp, so the oracle is the same; the bar is the
per-row bound of the accuracy statement in include/lse.h (e16_bound), special
values exactly, and the paper's own figure for the mean absolute error of its
16-bit variant (below 3e-3) on every workload.
"""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import (E16_BIAS, E16_OUT, LOG2E, compare, compare_e16, device_rows,
                          e16_bound, torch_view)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402

PAPER_MEAN_ABS_ERR = 3e-3  # FuseLSE16 at N = 128,256 (Sec. 4.3)


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bf16_values(lo: float, hi: float) -> np.ndarray:
    """Every positive bf16 value in [lo, hi], as float64."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)
    v = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    return v[(v >= lo) & (v <= hi)]


def test_packed_exponential_error():
    """What the bound assumes of the packed SFU instruction: a bf16 result at
    or below 2^a'', by less than a factor 1 - E16_OUT (it truncates), for every
    argument a'' on the bf16 grid in [-10, 0).  Rows [0, v] give
    lse = log(1 + t) with t the term of v; the maximum's own term is exactly 1."""
    _need_gpu()
    z = torch.tensor([[0.0, float("-inf")]], device="cuda")
    got, _ = L.lse_forward16(z)
    assert got.item() == 0.0  # 2^d truncates to exactly 1
    a = _bf16_values(2.0 ** -8, 10.0)
    v = (-a / LOG2E).astype(np.float32)
    # the kernel's argument: fl32(v log2 e + d), then bf16 (nearest even)
    arg = (v.astype(np.float64) * float(np.float32(LOG2E)) + float(np.float32(E16_BIAS)))
    arg = wl.f32_to_bf16_bits(arg.astype(np.float32)).astype(np.uint32) << np.uint32(16)
    exact = np.exp2(arg.view(np.float32).astype(np.float64))
    x = np.stack([np.zeros_like(v), v], axis=1)
    got, plan = L.lse_forward16(torch.from_numpy(x).cuda())
    t = np.expm1(got.cpu().numpy().astype(np.float64))
    eta = t / exact - 1.0
    # Reading error of t from an f32 lse: half an ulp of lse plus lg2 rounding.
    slack = 4e-7 * (1.0 + exact) / exact
    assert np.all(eta <= slack), (eta.max(), plan.as_dict())
    assert np.all(eta >= -E16_OUT - slack), (eta.min(), plan.as_dict())


@pytest.mark.parametrize("key", wl.ORDER)
def test_workloads(key):
    """Each row workload at full size, automatic plan."""
    _need_gpu()
    w = wl.WORKLOADS[key]
    x = wl.generate(key)
    want = oracle.lse(x, w.dtype)
    got, plan = L.lse_forward16(torch_view(x, w.dtype).cuda())
    torch.cuda.synchronize()
    s = compare_e16(got.cpu().numpy(), want, e16_bound(x, w.dtype, want))
    assert s["mean_abs_err"] < PAPER_MEAN_ABS_ERR, s
    # The truncation is compensated: no systematic offset of the row values
    # where arguments spread over the bf16 grid.  16-bit inputs can sit on a
    # coarse grid of their own (bf16 spacing is 4 near +-1000), so all their
    # arguments one step below the maximum round the same way and the offset
    # does not average out; there only the bound and the mean absolute error hold.
    if w.dtype == "f32":
        assert abs(s["mean_err"]) < PAPER_MEAN_ABS_ERR / 4, s


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_same_as_f32_path_on_exact_cases(dtype):
    """N = 1 gives x itself; constant rows (every argument 0, or the rounding
    residual of mu log2 e in the FFMA form, so every term is 1 in bf16) meet the
    f32 path's bar, not just the reduced-bit bound; N = 0 gives -inf; B = 0
    launches nothing."""
    _need_gpu()
    x = wl.random_rows(37, 1, dtype, seed=3)
    got, _ = L.lse_forward16(torch_view(x, dtype).cuda())
    want = oracle.lse(x, dtype)
    assert np.array_equal(got.cpu().numpy().astype(np.float64), want)
    c = np.repeat(wl.random_rows(40, 1, dtype, seed=4, scale=30.0), 1000, axis=1)
    for n in (1000, 40, 100000):  # sub-warp (FFMA form and not), CTA mappings
        cn = np.ascontiguousarray(c[:, :1].repeat(n, axis=1))
        got, _ = L.lse_forward16(torch_view(cn, dtype).cuda())
        compare(got.cpu().numpy(), oracle.lse(cn, dtype))
    e, _ = L.lse_forward16(torch.empty((5, 0), device="cuda",
                                       dtype={"f32": torch.float32, "bf16": torch.bfloat16,
                                              "f16": torch.float16}[dtype]))
    assert np.all(e.cpu().numpy() == -np.inf)
    b0, _ = L.lse_forward16(torch.empty((0, 9), device="cuda"))
    assert b0.numel() == 0


SPECIAL_ROWS = [
    [0.0, 1.0, float("nan"), 2.0],
    [float("inf"), 1.0, 2.0, 3.0],
    [float("inf"), float("nan"), 1.0, 1.0],
    [float("-inf")] * 4,
    [float("-inf"), float("-inf"), 5.0, float("-inf")],
    [float("inf"), float("-inf"), 0.0, 0.0],
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [4, 37, 1000, 70000])
def test_special_values(dtype, N):
    """NaN, +inf and all -inf rows exactly as lse_forward, on every mapping size."""
    _need_gpu()
    rng = np.random.default_rng(N)
    base = rng.normal(size=(len(SPECIAL_ROWS), N)).astype(np.float32)
    for i, r in enumerate(SPECIAL_ROWS):
        pos = rng.choice(N, size=min(4, N), replace=False)
        if all(v == float("-inf") for v in r):
            base[i, :] = -np.inf
        base[i, pos] = np.array(r[:len(pos)], dtype=np.float32)
    if dtype == "f32":
        x = base
    elif dtype == "f16":
        x = base.astype(np.float16)
    else:  # round the non-NaN values, then put the NaNs back as a quiet bf16 NaN
        x = wl.f32_to_bf16_bits(np.where(np.isnan(base), np.float32(0.0), base))
        x[np.isnan(base)] = 0x7FC0
    want = oracle.lse(x, dtype)
    got, _ = L.lse_forward16(torch_view(x, dtype).cuda())
    compare_e16(got.cpu().numpy(), want, e16_bound(x, dtype, want))


def _plans(rng, N, dtype, aligned, rs):
    eb = 4 if dtype == "f32" else 2
    epv = 16 // eb  # vector slots; rows off a 16-byte boundary peel a head and a tail slot
    slots = N // epv
    nvt = -(-N // epv) if aligned else N // epv + 2
    out = [None]
    if nvt <= 128:
        G = int(2 ** rng.integers(0, 6))
        if -(-nvt // G) <= 4 or (G >= 4 and -(-nvt // G) <= 8):
            out.append({"path": "subwarp", "lanes_per_row": G})
    elif nvt <= 256:
        out.append({"path": "subwarp", "lanes_per_row": 32})
    if slots >= 1:
        out.append({"path": "cta", "threads": int(32 * 2 ** rng.integers(0, 5))})
    if slots >= 2:
        out.append({"path": "split", "splits": int(rng.integers(2, min(slots, 40) + 1))})
    if aligned and rs == N and N * eb % 16 == 0 and 16 <= N * eb <= 128:
        out.append({"path": "rowtile"})
    return out


@pytest.mark.parametrize("seed", range(48))
def test_random_layouts_and_plans(seed):
    """Random dtype, shape, row stride, offset, value scale and every mapping."""
    _need_gpu()
    rng = np.random.default_rng(5000 + seed)
    dtype = ["f32", "bf16", "f16"][seed % 3]
    N = int(np.exp(rng.uniform(0, np.log(20000))))
    B = int(rng.integers(1, 200)) if N > 64 else int(rng.integers(1, 5000))
    rs = N + int(rng.choice([0, 0, 3, 8]))
    off = int(rng.choice([0, 0, 1]))
    scale = float(rng.choice([0.5, 4.0, 30.0]))
    shift = float(rng.choice([0.0, -40.0, 60.0]))
    x = wl.random_rows(B, N, dtype, seed=int(rng.integers(1 << 30)), scale=scale, shift=shift)
    _, xv = device_rows(x, dtype, row_stride=rs, offset=off)
    eb = 4 if dtype == "f32" else 2
    aligned = xv.data_ptr() % 16 == 0 and (rs * eb) % 16 == 0
    want = oracle.lse(x, dtype)
    bound = e16_bound(x, dtype, want)
    for plan in _plans(rng, N, dtype, aligned, rs):
        try:
            got, p = L.lse_forward16(xv, plan=plan)
        except L.LseError:
            if plan and plan["path"] == "rowtile":
                continue  # rows too few or misplaced for the bulk-copy mapping
            raise
        torch.cuda.synchronize()
        try:
            compare_e16(got.cpu().numpy(), want, bound)
        except AssertionError as exc:
            raise AssertionError(f"plan {p.as_dict()}: {exc}") from None


def test_reduced_bits_are_used():
    """The result differs from the f32-exponential path (same plan) on a row
    where bf16 rounding of the arguments shows, and stays within the bound."""
    _need_gpu()
    x = wl.random_rows(64, 4096, "f32", seed=11, scale=4.0)
    xt = torch.from_numpy(x).cuda()
    a, pa = L.lse_forward_plan(xt)
    b, pb = L.lse_forward16(xt)
    assert pa.as_dict()["path"] == pb.as_dict()["path"]
    want = oracle.lse(x, "f32")
    compare(a.cpu().numpy(), want)
    compare_e16(b.cpu().numpy(), want, e16_bound(x, "f32", want))
    assert not np.array_equal(a.cpu().numpy(), b.cpu().numpy())


def test_graph_capture():
    """Captured and replayed like lse_forward (split plans take pool scratch)."""
    _need_gpu()
    x = wl.random_rows(8, 300000, "bf16", seed=5)
    xt = torch_view(x, "bf16").cuda()
    out = torch.empty(8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        L.lse_forward16(xt, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _, p = L.lse_forward16(xt, out=out)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    want = oracle.lse(x, "bf16")
    compare_e16(out.cpu().numpy(), want, e16_bound(x, "bf16", want))
