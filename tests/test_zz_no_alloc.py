"""lse_forward_split_static: the entry point that allocates no device memory.

Some callers cannot allocate device memory while they run: a fixed memory
budget reserved up front, real-time loops where an allocator call may not
happen, or an allocator owned by another runtime.  For them the library keeps
the split-row partials in a fixed 1 MiB device array instead of per-call
scratch.  These tests call it through the C ABI and check it against
lse_forward (itself checked against the fp64 oracle elsewhere), twice in a
row, since consecutive calls reuse the same array.  The file sorts last so a
run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

from log_sum_exp_gb300 import workloads as wl
from lse_testutil import ATOL, RTOL, compare, torch_view

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


@pytest.mark.parametrize("key,B,N", [
    ("particles_16x16777216_f32", 4, 1 << 21),
    ("vocab_512x128256_f32", 64, None),
    ("vocab_8192x32000_bf16", 256, None),
])
def test_static_scratch_matches_lse_forward_twice(key, B, N):
    _need_gpu()
    w = wl.WORKLOADS[key]
    # Two different inputs through two consecutive calls: the second call
    # reuses the array the first one filled.
    xs = [wl.generate(key, B=B, N=N, seed=w.seed + k) for k in range(2)]
    outs = []
    for x in xs:
        xd = torch_view(x, w.dtype).cuda()
        got = _static(xd, w.dtype)
        want = L.lse_forward(xd)
        torch.cuda.synchronize()
        compare(got.cpu().numpy(), want.cpu().numpy().astype(np.float64), ATOL, RTOL)
        outs.append(got.cpu().numpy())
    assert not np.array_equal(outs[0], outs[1])


def test_static_scratch_special_values_and_unaligned_rows():
    _need_gpu()
    x = wl.random_rows(7, 5003, "f32", seed=5)
    x[1, 4000] = np.nan
    x[2, 17] = np.inf
    x[3, :] = -np.inf
    buf = torch.full((7 * 5005 + 3,), float("nan"), device="cuda")
    xv = buf[1:1 + 7 * 5005].view(7, 5005)[:, :5003]  # misaligned rows, padded stride
    xv.copy_(torch.from_numpy(x))
    for _ in range(2):
        got = _static(xv, "f32")
        want = L.lse_forward(xv)
        torch.cuda.synchronize()
        compare(got.cpu().numpy(), want.cpu().numpy().astype(np.float64), ATOL, RTOL)


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
