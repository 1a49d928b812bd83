"""lse_forward_split_static: the entry point that allocates no device memory.

Some callers cannot allocate device memory while they run: a fixed memory
budget reserved up front, real-time loops where an allocator call may not
happen, or an allocator owned by another runtime.  For them the library keeps
the split-row partials in a fixed 1 MiB device array instead of per-call
scratch.  These tests call it through the C ABI and compare every result with
the fp64 oracle at the parity bar (and with lse_forward as a second check).
Consecutive calls reuse the same array, so the calls come in sequences whose
shapes differ: a later call must never read a partial an earlier call left.
The file sorts last so a run that stops at the first failure has already run
every other test.
"""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import ATOL, RTOL, compare, device_rows, torch_view

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _static(xd, dtype):
    B, N = xd.shape
    out = torch.full((B,), float("nan"), dtype=torch.float32, device=xd.device)
    L.lse_forward_split_static_ptr(xd.data_ptr(), dtype, B, N, xd.stride(0), out.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    return out


def _check(xd, x, dtype):
    """The static entry point against the oracle and against lse_forward."""
    got = _static(xd, dtype)
    second = L.lse_forward(xd)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    compare(got, oracle.lse(x, dtype), ATOL, RTOL)
    compare(got, second.cpu().numpy().astype(np.float64), ATOL, RTOL)
    return got


@pytest.mark.parametrize("key,B,N", [
    ("particles_16x16777216_f32", 4, 1 << 21),
    ("vocab_512x128256_f32", 64, None),
    ("vocab_8192x32000_bf16", 256, None),
])
def test_static_scratch_matches_oracle_twice(key, B, N):
    _need_gpu()
    w = wl.WORKLOADS[key]
    # Two different inputs through two consecutive calls: the second call
    # reuses the array the first one filled.
    xs = [wl.generate(key, B=B, N=N, seed=w.seed + k) for k in range(2)]
    outs = [_check(torch_view(x, w.dtype).cuda(), x, w.dtype) for x in xs]
    assert not np.array_equal(outs[0], outs[1])


def test_static_scratch_large_call_then_small_call():
    """A call that fills the whole array with +inf and NaN partials, then a
    smaller call of another width: the second call's merge must read only the
    partials it wrote itself."""
    _need_gpu()
    B1, N1 = 65536, 64  # 65536 rows x 2 partials: the whole 1 MiB array
    x1 = np.full((B1, N1), np.inf, dtype=np.float32)
    x1[::2, 5] = np.nan
    _check(torch.from_numpy(x1).cuda(), x1, "f32")
    for B2, N2, seed in [(3, 4099, 1), (40, 1 << 15, 2), (1, 64, 3)]:
        x2 = wl.random_rows(B2, N2, "f32", seed=seed)
        _check(torch.from_numpy(x2).cuda(), x2, "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_static_scratch_special_values_and_unaligned_rows(dtype):
    _need_gpu()
    x = wl.random_rows(7, 5003, dtype, seed=5)
    if dtype == "f32":
        x[1, 4000], x[2, 17], x[3, :], x[4, 0], x[4, 5002] = np.nan, np.inf, -np.inf, np.inf, np.nan
    else:
        bits = {"bf16": (0x7FC0, 0x7F80, 0xFF80), "f16": (0x7E00, 0x7C00, 0xFC00)}[dtype]
        xb = x.view(np.uint16)
        xb[1, 4000], xb[2, 17], xb[3, :] = bits[0], bits[1], bits[2]
        xb[4, 0], xb[4, 5002] = bits[1], bits[0]
    # Rows one element past a 16-byte boundary, stride padded by two elements.
    _, xv = device_rows(x, dtype, row_stride=5005, offset=1)
    for _ in range(2):
        _check(xv, x, dtype)


def test_static_scratch_allocates_no_device_memory():
    """After a first call (which looks the array's address up), further calls
    leave the device's free memory unchanged."""
    _need_gpu()
    x = wl.random_rows(64, 1 << 16, "f32", seed=9)
    xd = torch.from_numpy(x).cuda()
    outs = [torch.empty(64, dtype=torch.float32, device="cuda") for _ in range(8)]
    sh = torch.cuda.current_stream().cuda_stream
    L.lse_forward_split_static_ptr(xd.data_ptr(), "f32", 64, 1 << 16, 1 << 16, outs[0].data_ptr(), sh)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for o in outs:
        L.lse_forward_split_static_ptr(xd.data_ptr(), "f32", 64, 1 << 16, 1 << 16, o.data_ptr(), sh)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    want = oracle.lse(x, "f32")
    for o in outs:
        compare(o.cpu().numpy(), want, ATOL, RTOL)


def test_static_scratch_rejects_too_many_rows():
    _need_gpu()
    x = torch.zeros((65537, 64), device="cuda")
    out = torch.empty(65537, device="cuda")
    with pytest.raises(L.LseError) as e:
        L.lse_forward_split_static_ptr(x.data_ptr(), "f32", 65537, 64, 64, out.data_ptr())
    assert e.value.status == 1
    # Rows too short to split are rejected too.
    with pytest.raises(L.LseError):
        L.lse_forward_split_static_ptr(x.data_ptr(), "f32", 4, 4, 64, out.data_ptr())
