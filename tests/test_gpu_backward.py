"""GPU parity of lse_backward against the fp64 oracle:
dx[b, n] = grad[b] * exp(x[b, n] - lse[b]).

The GPU receives the oracle's row values rounded to f32 (as a saved forward
output would be), the oracle keeps them in fp64.  Per-element bar, from the
f32 arithmetic of the kernel (ex2.approx ~2^-22, rounding of lse and of
x - lse at 2^-24 of their magnitudes) and the output rounding of the dtype:
    |d| <= |g| * 1e-37 + |ref| * (2^-21 + 2^-23 (|lse| + |x - lse|) + q)
with q = 0 (f32), 2^-8 (bf16), 2^-11 (f16) plus 2^-24 absolute for f16
subnormals.  NaN and +-inf must match exactly.
"""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import canary_array, compare_backward, torch_view

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402

def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _decode(x, dtype):
    return oracle.decode(x, dtype).reshape(x.shape)


def _check(got_raw, x, dtype, lse64, g, want):
    return compare_backward(_decode(got_raw, dtype), _decode(x, dtype), dtype, lse64, g, want)


def _run(x, dtype, g, row_stride=None, offset=0, dx_row_stride=None, dx_offset=0, inplace=False):
    """Call lse_backward on device copies inside NaN-canaried buffers."""
    B, N = x.shape
    lse64 = oracle.lse(x, dtype)
    want = oracle.backward(x, lse64, g, dtype)
    rs = N if row_stride is None else row_stride
    ds = rs if inplace else (N if dx_row_stride is None else dx_row_stride)
    xh = canary_array(offset + B * rs + 32, dtype)
    xh[offset:offset + B * rs].reshape(B, rs)[:, :N] = x if dtype == "f32" else x.view(np.uint16)
    xbuf = torch_view(xh, dtype).cuda()
    if inplace:
        dbuf, doff = xbuf, offset
    else:
        dbuf = torch_view(canary_array(dx_offset + B * ds + 32, dtype), dtype).cuda()
        doff = dx_offset
    eb = 4 if dtype == "f32" else 2
    lse_d = torch.from_numpy(lse64.astype(np.float32)).cuda()
    g_d = torch.from_numpy(g.astype(np.float32)).cuda()
    L.lse_backward_ptr(xbuf.data_ptr() + offset * eb, dtype, B, N, rs, lse_d.data_ptr(),
                       g_d.data_ptr(), dbuf.data_ptr() + doff * eb, ds)
    torch.cuda.synchronize()
    host = dbuf.cpu()
    raw = host.numpy() if dtype == "f32" else host.view(torch.int16).numpy().view(np.uint16)
    body = raw[doff:doff + B * ds].reshape(B, ds)
    got = np.ascontiguousarray(body[:, :N])
    # Canaries: nothing outside the [B, N] block of dx may change.
    mask = np.ones(raw.shape, bool)
    mask[doff:doff + B * ds] = False
    pad = np.ones((B, ds), bool)
    pad[:, :N] = False
    outside = np.concatenate([raw[mask], body[pad]])
    if dtype == "f32":
        assert np.all(np.isnan(outside)), "write outside dx rows"
    else:
        assert np.all(outside == (0x7FC0 if dtype == "bf16" else 0x7E00)), "write outside dx rows"
    return got, lse64, want


@pytest.mark.parametrize("key,B,N", [
    ("vocab_512x128256_f32", 32, None),
    ("vocab_8192x32000_bf16", 256, None),
    ("short_1048576x32_f32", 100000, None),
    ("particles_16x16777216_f32", 2, 1 << 21),
    ("small_64x4096_f32", None, None),
])
def test_workload_backward(key, B, N):
    _need_gpu()
    w = wl.WORKLOADS[key]
    x = wl.generate(key, B=B, N=N)
    g = np.random.default_rng(w.index).normal(0, 2, x.shape[0])
    got, lse64, want = _run(x, w.dtype, g)
    r = _check(got, x, w.dtype, lse64, g, want)
    print(key, "max err / tol", r)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8, 9, 12, 15, 16, 17, 31, 32, 33, 1000, 4097,
                               20001])
def test_backward_edge_shapes(dtype, N):
    _need_gpu()
    B = 7
    x = wl.random_rows(B, N, dtype, seed=200 + N, scale=4.0)
    if N >= 3:
        xi = x.view(np.uint16) if dtype != "f32" else x
        ninf = {"f32": -np.inf, "bf16": 0xFF80, "f16": 0xFC00}[dtype]
        nan = {"f32": np.nan, "bf16": 0x7FC0, "f16": 0x7E00}[dtype]
        xi[2, :] = ninf           # lse = -inf: NaN gradient
        xi[3, N // 2] = nan       # NaN row
        xi[4, ::2] = ninf         # zeros in the gradient
    g = np.random.default_rng(N).normal(0, 3, B)
    g[5] = 0.0
    eb = 4 if dtype == "f32" else 2
    # Element slots where x and dx rows sit at different offsets from a 16-byte
    # boundary; vectors with a peeled head and tail where they share it.
    layouts = [dict(), dict(row_stride=N + 8, dx_row_stride=N + 8), dict(row_stride=N + 3),
               dict(offset=1), dict(dx_offset=1), dict(inplace=True),
               dict(offset=1, dx_offset=1), dict(row_stride=N + 3, dx_row_stride=N + 3),
               dict(offset=3, dx_offset=3 + 16 // eb, row_stride=N + 1,
                    dx_row_stride=N + 1 + 16 // eb),
               dict(inplace=True, offset=1, row_stride=N + 1)]
    for lay in layouts:
        got, lse64, want = _run(x, dtype, g, **lay)
        try:
            _check(got, x, dtype, lse64, g, want)
        except AssertionError as e:
            raise AssertionError(f"layout {lay}: {e}") from None


def test_backward_tensor_api_and_bad_args():
    _need_gpu()
    x = torch.randn(8, 100, device="cuda")
    lse = L.lse_forward(x)
    g = torch.ones(8, device="cuda")
    dx = L.lse_backward(x, lse, g)
    assert torch.allclose(dx.sum(dim=1), g, rtol=1e-5)
    with pytest.raises(L.LseError):
        L.lse_backward_ptr(x.data_ptr(), "f32", 8, 100, 100, lse.data_ptr(), g.data_ptr(),
                           dx.data_ptr(), 99)
    with pytest.raises(L.LseError):
        L.lse_backward_ptr(x.data_ptr(), "f32", 8, 100, 100, 0, g.data_ptr(), dx.data_ptr(), 100)
    with pytest.raises(L.LseError):
        L.lse_backward_ptr(x.data_ptr(), "f32", 8, 100, 100, lse.data_ptr(), g.data_ptr(),
                           dx.data_ptr() + 2, 100)


@pytest.mark.parametrize("seed", range(40))
def test_backward_random_layouts(seed):
    """Random dtype, shape, offsets and strides of x and dx: element slots,
    16-byte vectors, or vectors with a peeled head and tail, against the
    oracle, with nothing written outside dx's rows."""
    _need_gpu()
    rng = np.random.default_rng(7000 + seed)
    dtype = ["f32", "bf16", "f16"][seed % 3]
    N = int(np.exp(rng.uniform(0, np.log(30000))))
    B = int(rng.integers(1, 64)) if N > 256 else int(rng.integers(1, 3000))
    off = int(rng.choice([0, 1, 2, 5]))
    rs = N + int(rng.choice([0, 0, 1, 3, 8]))
    if rng.random() < 0.5:  # dx at the same offset from a 16-byte boundary as x
        eb = 4 if dtype == "f32" else 2
        lay = dict(offset=off, row_stride=rs, dx_offset=off + int(rng.choice([0, 16 // eb])),
                   dx_row_stride=rs + int(rng.choice([0, 16 // eb])))
    else:
        lay = dict(offset=off, row_stride=rs, dx_offset=int(rng.choice([0, 1, 3])),
                   dx_row_stride=N + int(rng.choice([0, 1, 2])))
    x = wl.random_rows(B, N, dtype, seed=int(rng.integers(1 << 30)),
                       scale=float(rng.choice([0.5, 4.0, 20.0])))
    g = rng.normal(0, 2, B)
    got, lse64, want = _run(x, dtype, g, **lay)
    try:
        _check(got, x, dtype, lse64, g, want)
    except AssertionError as e:
        raise AssertionError(f"B={B} N={N} layout {lay}: {e}") from None


@pytest.mark.parametrize("dtype,B,N,off", [("bf16", 100003, 37, 0), ("f32", 30001, 129, 1),
                                           ("f16", 4099, 1001, 3), ("f32", 3, 8, 1),
                                           ("bf16", 1, 8, 5)])
def test_backward_flat_rows(dtype, B, N, off):
    """Back-to-back rows whose starts are not all on a 16-byte boundary: the
    whole block streamed as one array of vectors spanning row ends, with many
    CTAs striding through it (and in place)."""
    _need_gpu()
    x = wl.random_rows(B, N, dtype, seed=B + N, scale=6.0)
    g = np.random.default_rng(N).normal(0, 2, B)
    for lay in (dict(offset=off, dx_offset=off), dict(inplace=True, offset=off)):
        got, lse64, want = _run(x, dtype, g, **lay)
        try:
            _check(got, x, dtype, lse64, g, want)
        except AssertionError as e:
            raise AssertionError(f"layout {lay}: {e}") from None
