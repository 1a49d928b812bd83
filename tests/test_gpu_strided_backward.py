"""GPU parity of lse_backward_strided (the gradient of the value over a
non-last dimension) against the fp64 oracle:
dx[a, r, c] = grad[a, c] * exp(x[a*sa + r*sr + c] - lse[a, c])."""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import NAN_BITS, canary_array, compare_backward, torch_view

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _raw(t, dtype):
    h = t.cpu()
    return h.numpy() if dtype == "f32" else h.view(torch.int16).numpy().view(np.uint16)


def _check_canaries(raw, keep, dtype):
    outside = raw[~keep]
    if dtype == "f32":
        assert np.all(np.isnan(outside)), "write outside dx"
    else:
        assert np.all(outside == NAN_BITS[dtype]), "write outside dx"


def run(x3, dtype, pad_r=0, pad_a=0, offset=0, inplace=False, seed=0):
    """x3: [A, R, C] raw elements.  Places x (and dx) in NaN-canaried buffers with
    the given padding, calls lse_backward_strided, checks against the oracle."""
    A, R, C = x3.shape
    bits = x3.view(np.uint16) if dtype == "f16" else x3  # f16 rows come as float16 values
    sr = C + pad_r
    sa = R * sr + pad_a
    span = (A - 1) * sa + (R - 1) * sr + C
    flat = canary_array(offset + span + 32, dtype)
    keep = np.zeros(flat.size, bool)
    for a in range(A):
        for r in range(R):
            lo = offset + a * sa + r * sr
            flat[lo:lo + C] = bits[a, r]
            keep[lo:lo + C] = True
    lse64 = oracle.lse_strided(np.ascontiguousarray(x3).reshape(-1), dtype, A, R, C, R * C, C)
    g = np.random.default_rng(seed).normal(0, 1.5, (A, C))
    want = oracle.backward_strided(np.ascontiguousarray(x3).reshape(-1), dtype, A, R, C, R * C, C,
                                   lse64, g)
    eb = 4 if dtype == "f32" else 2
    xbuf = torch_view(flat, dtype).cuda()
    if inplace:
        dbuf, doff, dsa, dsr = xbuf, offset, sa, sr
    else:
        dbuf = torch_view(canary_array(A * R * C + 32, dtype), dtype).cuda()
        doff, dsa, dsr = 0, R * C, C
    lse_d = torch.from_numpy(lse64.astype(np.float32)).cuda()
    g_d = torch.from_numpy(g.astype(np.float32)).cuda()
    L.lse_backward_strided_ptr(xbuf.data_ptr() + offset * eb, dtype, A, R, C, sa, sr,
                               lse_d.data_ptr(), g_d.data_ptr(), dbuf.data_ptr() + doff * eb,
                               dsa, dsr, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    raw = _raw(dbuf, dtype)
    if inplace:
        got = np.stack([np.stack([raw[offset + a * sa + r * sr:offset + a * sa + r * sr + C]
                                  for r in range(R)]) for a in range(A)])
        _check_canaries(raw, keep, dtype)
    else:
        got = raw[:A * R * C].reshape(A, R, C)
        dk = np.zeros(raw.size, bool)
        dk[:A * R * C] = True
        _check_canaries(raw, dk, dtype)
    dec = lambda v: oracle.decode(np.ascontiguousarray(v), dtype).reshape(v.shape)  # noqa: E731
    rows = lambda v: np.ascontiguousarray(v.transpose(0, 2, 1)).reshape(A * C, R)  # noqa: E731
    return compare_backward(rows(dec(got)), rows(dec(x3)), dtype, lse64.reshape(-1),
                            g.reshape(-1), rows(want))


SHAPES = [(3, 37, 21), (4, 64, 1024), (2, 300, 136), (1, 5, 7), (1, 1000, 1), (5, 1, 64),
          (2, 2049, 40)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{a}x{r}x{c}" for a, r, c in SHAPES])
def test_shapes_and_layouts(dtype, shape):
    _need_gpu()
    A, R, C = shape
    x3 = wl.random_rows(A * R, C, dtype, seed=A * R + C, scale=4.0).reshape(A, R, C)
    eb = 4 if dtype == "f32" else 2
    for pad_r, pad_a, offset in ((0, 0, 0), (16 // eb, 8, 0), (3, 5, 0), (0, 0, 1)):
        run(x3, dtype, pad_r, pad_a, offset, seed=pad_r + offset)
    run(x3, dtype, inplace=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_narrow_column_tiles(dtype):
    """Narrow C: one-warp units of 16- or 8-lane tiles, two or four side by
    side in a warp (the later groups of lanes take the next units, possibly of
    the next a); aligned, padded and element layouts, and in place."""
    _need_gpu()
    eb = 4 if dtype == "f32" else 2
    for A, R, C in ((37, 64, 64), (100, 9, 128), (20, 33, 40), (7, 70, 200), (3, 5, 384),
                    (1, 3, 16), (513, 2, 8), (65, 4, 32)):
        x3 = wl.random_rows(A * R, C, dtype, seed=A + R + C, scale=4.0).reshape(A, R, C)
        for pad_r, pad_a, offset in ((0, 0, 0), (16 // eb, 8, 0), (3, 5, 0), (0, 0, 1)):
            run(x3, dtype, pad_r, pad_a, offset, seed=A + pad_r + offset)
        run(x3, dtype, inplace=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_special_values(dtype):
    _need_gpu()
    A, R, C = 2, 33, 64
    x3 = wl.random_rows(A * R, C, "f32", seed=8, scale=3.0).reshape(A, R, C)
    x3[0, :, 3] = -np.inf          # all -inf column: lse -inf, dx NaN
    x3[0, 5, 4] = np.nan           # NaN column
    x3[1, 7, 5] = np.inf           # +inf column
    x3[1, ::3, 6] = -np.inf        # some -inf: those dx are 0
    if dtype == "bf16":
        x3 = wl.f32_to_bf16_bits(np.where(np.isnan(x3), np.float32(0), x3))
        x3[0, 5, 4] = NAN_BITS["bf16"]
    run(x3, dtype)


def test_sum_layer_workload():
    """The full sum-layer workload (512 x 64 x 1024 f32)."""
    _need_gpu()
    cw = wl.COLUMN_WORKLOADS["pcsum_512x64x1024_f32"]
    run(wl.generate_columns(cw.key), "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dim", [0, 1])
def test_logsumexp_autograd_other_dims(dtype, dim):
    """logsumexp over a non-last dimension is differentiable through
    lse_backward_strided: x.grad against the oracle."""
    _need_gpu()
    A, R, C = 6, 40, 48
    x = wl.random_rows(A * R, C, dtype, seed=dim + 3, scale=5.0).reshape(A, R, C)
    if dim == 0:  # reduce over the first dimension: [1, A, R*C] in oracle terms
        shape3 = (1, A, R * C)
    else:
        shape3 = (A, R, C)
    xd = torch_view(x.reshape(-1), dtype).cuda().reshape(A, R, C).requires_grad_(True)
    y = L.logsumexp(xd, dim=dim)
    w = np.random.default_rng(dim).normal(size=y.shape).astype(np.float32)
    (y * torch.from_numpy(w).cuda()).sum().backward()
    a3, r3, c3 = shape3
    lse64 = oracle.lse_strided(x.reshape(-1), dtype, a3, r3, c3, r3 * c3, c3)
    want = oracle.backward_strided(x.reshape(-1), dtype, a3, r3, c3, r3 * c3, c3, lse64,
                                   w.reshape(a3, c3).astype(np.float64))
    dec = lambda v: oracle.decode(np.ascontiguousarray(v), dtype).reshape(v.shape)  # noqa: E731
    got = dec(_raw(xd.grad, dtype)).reshape(a3, r3, c3)
    rows = lambda v: np.ascontiguousarray(v.transpose(0, 2, 1)).reshape(a3 * c3, r3)  # noqa: E731
    compare_backward(rows(got), rows(dec(x).reshape(a3, r3, c3)), dtype, lse64.reshape(-1),
                     w.reshape(-1).astype(np.float64), rows(want))
