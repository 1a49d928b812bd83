"""GPU parity of lse_forward_strided (the value over a non-last dimension)
against the fp64 oracle: out[a, c] = log sum_r exp(x[a*sa + r*sr + c])."""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import canary_array, compare, torch_view

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_strided(x3, dtype, pad_r=0, pad_c=0, pad_a=0, offset=0, plan=None):
    """Place x [A, R, C] in a NaN-canaried buffer with padded strides and run."""
    A, R, C = x3.shape
    sr = C + pad_c
    sa = R * sr + pad_a + pad_r * sr
    total = offset + max(A, 1) * sa + 64
    host = canary_array(total, dtype)
    for a in range(A):
        blk = host[offset + a * sa: offset + a * sa + R * sr].reshape(R, sr)
        blk[:, :C] = x3[a] if dtype == "f32" else x3[a].view(np.uint16)
    buf = torch_view(host, dtype).cuda()
    eb = 4 if dtype == "f32" else 2
    out = torch.full((A * C + 16,), float("nan"), device="cuda")
    L.lse_forward_strided_ptr(buf.data_ptr() + offset * eb, dtype, A, R, C, sa, sr, out.data_ptr(),
                              torch.cuda.current_stream().cuda_stream, plan)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.all(np.isnan(o[A * C:])), "write past out[A*C-1]"
    want = oracle.lse_strided(host[offset:], dtype, A, R, C, sa, sr)
    return o[:A * C].reshape(A, C), want


@pytest.mark.parametrize("key", list(wl.COLUMN_WORKLOADS))
def test_column_workloads(key):
    _need_gpu()
    x = wl.generate_columns(key)
    got, want = run_strided(x, "f32")
    print(key, compare(got, want))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("A,R,C", [(1, 1, 1), (1, 5, 3), (2, 1, 64), (3, 7, 8), (2, 33, 129),
                                   (5, 64, 1000), (1, 300, 256), (1, 1000, 17), (4, 2, 4096)])
def test_strided_edge_shapes(dtype, A, R, C):
    _need_gpu()
    x = wl.random_rows(A * R, C, dtype, seed=A * 1000 + R * 10 + C, scale=5.0).reshape(A, R, C)
    if R >= 3 and C >= 4:
        xi = x.view(np.uint16) if dtype != "f32" else x
        xi[0, :, 1] = {"f32": -np.inf, "bf16": 0xFF80, "f16": 0xFC00}[dtype]
        xi[0, R // 2, 2] = {"f32": np.nan, "bf16": 0x7FC0, "f16": 0x7E00}[dtype]
        xi[A - 1, R - 1, 3] = {"f32": np.inf, "bf16": 0x7F80, "f16": 0x7C00}[dtype]
    for lay in (dict(), dict(pad_c=8), dict(pad_c=3), dict(offset=1), dict(pad_a=8, pad_r=1)):
        for path, wt in (("auto", 0), ("columns_warp", 0), ("columns_cta", 2), ("columns_cta", 4),
                         ("columns_cta", 8)):
            for splits in (0, 1, 2, 3):
                if splits > R:
                    continue
                plan = {"path": path, "splits": splits, "lanes_per_row": wt}
                got, want = run_strided(x, dtype, plan=plan, **lay)
                try:
                    compare(got, want)
                except AssertionError as e:
                    raise AssertionError(f"layout {lay} plan {plan}: {e}") from None


def test_strided_degenerate():
    _need_gpu()
    out = torch.full((6,), 7.0, device="cuda")
    x = torch.zeros(16, device="cuda")
    p = L.lse_forward_strided_ptr(x.data_ptr(), "f32", 2, 0, 3, 0, 0, out.data_ptr())
    torch.cuda.synchronize()
    assert np.all(out.cpu().numpy() == -np.inf) and p.as_dict()["path"] == "empty"
    L.lse_forward_strided_ptr(x.data_ptr(), "f32", 0, 4, 3, 12, 3, out.data_ptr())  # no-op
    with pytest.raises(L.LseError):
        L.lse_forward_strided_ptr(x.data_ptr(), "f32", 1, 4, 3, 12, -3, out.data_ptr())
    with pytest.raises(L.LseError):
        L.lse_forward_strided_ptr(x.data_ptr(), "f32", 1, 4, 3, 12, 3, out.data_ptr(),
                                  plan={"splits": 5})
    with pytest.raises(L.LseError):
        L.lse_forward_strided_ptr(x.data_ptr(), "f32", 1, 4, 3, 12, 3, out.data_ptr(),
                                  plan={"path": "split"})


def _oracle_over_dim(x, dtype, d):
    """The oracle's value over dimension d of a contiguous array, as [outer, inner]."""
    shape = x.shape
    outer = int(np.prod(shape[:d], dtype=np.int64))
    inner = int(np.prod(shape[d + 1:], dtype=np.int64))
    R = shape[d]
    out = oracle.lse_strided(np.ascontiguousarray(x).reshape(-1), dtype, outer, R, inner,
                             R * inner, inner)
    return out.reshape(shape[:d] + shape[d + 1:])


def test_logsumexp_any_dim():
    _need_gpu()
    x = wl.random_rows(6 * 40, 33, "f32", seed=9, scale=6.0).reshape(6, 40, 33)
    xd = torch.from_numpy(x).cuda()
    for dim in (0, 1, 2, -1):
        got = L.logsumexp(xd, dim=dim).cpu().numpy()
        compare(got, _oracle_over_dim(x, "f32", dim % 3))
        kd = L.logsumexp(xd, dim=dim, keepdim=True)
        assert kd.shape == torch.logsumexp(torch.from_numpy(x), dim=dim, keepdim=True).shape


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_logsumexp_autograd_last_dim(dtype):
    """y = logsumexp(x, -1) is differentiable: x.grad = g * exp(x - y) through
    lse_backward, checked against the oracle's backward; keepdim and a 3-D x."""
    _need_gpu()
    from lse_testutil import compare_backward

    x = wl.random_rows(6 * 50, 300, dtype, seed=12, scale=5.0)
    w = np.random.default_rng(3).normal(size=300).astype(np.float32)
    for shape, keepdim in (((300, 300), False), ((6, 50, 300), True)):
        xd = torch_view(x, dtype).cuda().reshape(shape).requires_grad_(True)
        y = L.logsumexp(xd, dim=-1, keepdim=keepdim)
        lse64 = oracle.lse(x, dtype)
        compare(y.detach().cpu().numpy().reshape(-1), lse64)
        (y.reshape(-1) * torch.from_numpy(w).cuda()).sum().backward()
        assert xd.grad.dtype == xd.dtype and xd.grad.shape == xd.shape
        raw = xd.grad.reshape(300, 300).cpu()
        raw = raw.numpy() if dtype == "f32" else raw.view(torch.int16).numpy().view(np.uint16)
        dec = lambda a: oracle.decode(a, dtype).reshape(a.shape)  # noqa: E731
        compare_backward(dec(raw), dec(x), dtype, lse64, w.astype(np.float64),
                         oracle.backward(x, lse64, w.astype(np.float64), dtype))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_columns_extreme_magnitudes(dtype):
    """Columns whose maximum is beyond 2^126 (the one-FFMA term form would
    overflow its shift; the fold falls back to the two-step form for the
    whole warp) beside ordinary columns, and the special values, on every
    column plan."""
    _need_gpu()
    big = 3.0e38
    cols = [[big, big], [-big, big], [big, -np.inf], [-big, -big], [1e-40, -1e-40],
            [-1e30, -1e30 + 1e24], [88.7, 88.7, 88.7], [-103.0, -103.0], [np.inf, -np.inf],
            [np.nan, -np.inf], [1.0, 2.0, 3.0], [2.0 ** 127, 2.0 ** 126]]
    R = 40
    rng = np.random.default_rng(7)
    C = 256
    base = rng.normal(0, 3, (2, R, C)).astype(np.float32)
    for k, col in enumerate(cols):
        c = (k * 37) % C
        base[:, :, c] = -np.inf
        base[:, :len(col), c] = col
    if dtype == "f32":
        x = base
    else:
        x = wl.f32_to_bf16_bits(np.where(np.isnan(base), np.float32(0.0), base))
        x[np.isnan(base)] = 0x7FC0
    for plan in (None, {"path": "columns_warp"}, {"path": "columns_cta", "lanes_per_row": 2},
                 {"path": "columns_cta", "lanes_per_row": 8}, {"path": "columns_warp", "splits": 3}):
        got, want = run_strided(x, dtype, plan=plan)
        try:
            compare(got, want)
        except AssertionError as e:
            raise AssertionError(f"plan {plan}: {e}") from None


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("offset", [0, 1])
def test_columns_inf_between_shifts(dtype, offset):
    """Columns where +inf arrives between runs of values far apart (the
    16-bit fold keeps a lazy shift per column: once a column has met +inf its
    shift must not move again), +inf first or last, two +inf, NaN beside
    +inf; aligned and realigned (offset) tiles, every column plan."""
    _need_gpu()
    R, C = 96, 40
    rng = np.random.default_rng(11)
    x = rng.normal(0, 2, (2, R, C)).astype(np.float32)
    x[:, :, 0] = 100.0
    x[:, 30, 0] = np.inf                                # finite, +inf, finite
    x[:, :40, 1] = -100.0
    x[:, 40, 1] = np.inf
    x[:, 41:, 1] = 100.0                                # low, +inf, high
    x[:, 0, 2] = np.inf                                 # +inf first
    x[:, R - 1, 3] = np.inf                             # +inf last
    x[:, 5, 4] = np.inf
    x[:, 70, 4] = np.inf                                # twice
    x[:, 10, 5] = np.nan
    x[:, 60, 5] = np.inf                                # NaN and +inf
    x[:, :, 6] = -np.inf
    x[:, 50, 6] = np.inf                                # only -inf and +inf
    if dtype == "f32":
        xx = x
    elif dtype == "f16":
        xx = x.astype(np.float16)
    else:
        xx = wl.f32_to_bf16_bits(np.where(np.isnan(x), np.float32(0.0), x))
        xx[np.isnan(x)] = 0x7FC0
    for plan in (None, {"path": "columns_warp"}, {"path": "columns_cta", "lanes_per_row": 2},
                 {"path": "columns_cta", "lanes_per_row": 4}, {"path": "columns_cta", "lanes_per_row": 8},
                 {"path": "columns_warp", "splits": 3}):
        got, want = run_strided(xx, dtype, offset=offset, plan=plan)
        try:
            compare(got, want)
        except AssertionError as e:
            raise AssertionError(f"plan {plan}: {e}") from None


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_columns_narrow_tiles(dtype):
    """Narrow C: tiles of 16 or 8 lanes, two or four per warp (the later
    groups of lanes fold the next (a, tile) units, possibly of the next a),
    walked by one warp or shared by 2 or 4 (merged lane by lane).  Special
    values in columns of several groups; aligned and element layouts; the
    warp and CTA paths forced and automatic; row splits."""
    _need_gpu()
    for A, R, C in ((37, 64, 64), (100, 9, 128), (20, 33, 40), (7, 70, 200), (3, 5, 384), (1, 3, 16),
                    (513, 2, 8), (65, 4, 32), (9, 17, 192)):
        x = wl.random_rows(A * R, C, dtype, seed=A + R + C, scale=5.0).reshape(A, R, C)
        xi = x.view(np.uint16) if dtype != "f32" else x
        nan, pinf, ninf = {"f32": (np.nan, np.inf, -np.inf), "bf16": (0x7FC0, 0x7F80, 0xFF80),
                           "f16": (0x7E00, 0x7C00, 0xFC00)}[dtype]
        if C >= 4:
            xi[A - 1, :, C - 1] = ninf
            xi[A - 1, R // 2, C - 2] = nan
            xi[0, R - 1, C // 2] = pinf
            xi[0, :, 0] = ninf
            xi[0, 0, 0] = 0
        for lay in (dict(), dict(pad_c=3), dict(offset=1)):
            for plan in (None, {"path": "columns_warp"}, {"path": "columns_warp", "splits": 2},
                         {"path": "columns_cta", "lanes_per_row": 2},
                         {"path": "columns_cta", "lanes_per_row": 4, "splits": 2}):
                if plan and plan.get("splits", 0) > R:
                    continue
                got, want = run_strided(x, dtype, plan=plan, **lay)
                try:
                    compare(got, want)
                except AssertionError as e:
                    raise AssertionError(f"shape {(A, R, C)} layout {lay} plan {plan}: {e}") from None


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_columns_short_reductions(dtype):
    """R <= 8 rows of 16-byte column vectors: a thread per vector folds all R
    rows (automatic there, and forced).  Every R, special values (an all -inf
    column, NaN, +inf, -inf among finite values), padded strides that keep
    the vector layout, and an output off a 16-byte boundary (scalar stores)."""
    _need_gpu()
    eb = 4 if dtype == "f32" else 2
    epv = 16 // eb
    for R in range(1, 9):
        for A, C in ((3, 8 * epv), (37, 2 * epv), (1, 64 * epv)):
            x = wl.random_rows(A * R, C, dtype, seed=R * 100 + A + C, scale=5.0).reshape(A, R, C)
            xi = x.view(np.uint16) if dtype != "f32" else x
            ninf, pinf, nan = {"f32": (-np.inf, np.inf, np.nan), "bf16": (0xFF80, 0x7F80, 0x7FC0),
                               "f16": (0xFC00, 0x7C00, 0x7E00)}[dtype]
            xi[0, :, 1] = ninf                   # all -inf
            xi[A - 1, R - 1, C - 1] = nan
            xi[A // 2, 0, C // 2] = pinf
            if R > 1:
                xi[0, R // 2, 3] = ninf          # -inf among finite values
            for lay in (dict(), dict(pad_c=epv), dict(pad_a=2 * epv, pad_r=1)):
                for plan in (None, {"path": "columns_short"}):
                    got, want = run_strided(x, dtype, plan=plan, **lay)
                    try:
                        compare(got, want)
                    except AssertionError as e:
                        raise AssertionError(f"R={R} A={A} C={C} layout {lay} plan {plan}: {e}") from None
            # out off a 16-byte boundary
            xd = torch_view(np.ascontiguousarray(x).reshape(-1) if dtype == "f32"
                            else np.ascontiguousarray(xi).reshape(-1), dtype).cuda()
            out = torch.full((A * C + 8,), float("nan"), device="cuda")
            p = L.lse_forward_strided_ptr(xd.data_ptr(), dtype, A, R, C, R * C, C, out.data_ptr() + 4,
                                          torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert p.as_dict()["path"] == "columns_short"
            o = out.cpu().numpy()
            assert np.isnan(o[0]) and np.all(np.isnan(o[A * C + 1:])), "write outside out"
            want = oracle.lse_strided(np.ascontiguousarray(x).reshape(-1), dtype, A, R, C, R * C, C)
            compare(o[1:A * C + 1].reshape(A, C), want)


def test_columns_short_rejects_other_layouts():
    _need_gpu()
    x = torch.zeros(4, 9, 64, device="cuda")
    with pytest.raises(L.LseError):
        L.lse_forward_strided_ptr(x.data_ptr(), "f32", 4, 9, 64, 9 * 64, 64,
                                  torch.empty(256, device="cuda").data_ptr(),
                                  torch.cuda.current_stream().cuda_stream, {"path": "columns_short"})
    with pytest.raises(L.LseError):  # C = 63: element layout
        L.lse_forward_strided_ptr(x.data_ptr(), "f32", 4, 4, 63, 4 * 63, 63,
                                  torch.empty(256, device="cuda").data_ptr(),
                                  torch.cuda.current_stream().cuda_stream, {"path": "columns_short"})
