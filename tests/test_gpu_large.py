"""Sizes past the 32-bit limits, against the fp64 oracle: rows that start more
than 4 GiB into the buffer, a row longer than 2^31 elements, and column strides
beyond 4 GiB (every offset in the kernels is 64-bit).

Expected values come from the oracle on the rows themselves, or, for the long
row, on the one seeded block it is made of: k copies of a block followed by
its first r elements have the row value log(k e^{LSE(block)} + e^{LSE(block[:r])})
by split associativity (a property the oracle is pinned to), and every other
expected quantity (token log-probability, gradient, the 16-bit bound) is the
oracle's value for the block element at the same position modulo the block.
"""
import gc

import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import (ATOL, RTOL, compare, compare_backward, compare_e16, compare_logprob,
                          e16_bound, e16_error_sum, torch_view)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402

GIB = 1 << 30


def _need(bytes_needed: int):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < bytes_needed + GIB:
        pytest.skip(f"needs {bytes_needed / GIB:.1f} GiB of free device memory")


def _tdt(dtype):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]


def _release():
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [64, 4096])
def test_row_offsets_beyond_4gib(dtype, N):
    """Four rows about 2 GiB apart (rows 2 and 3 start past 4 GiB): row value
    on every mapping that takes strided rows, token log-probability, 16-bit
    exponentials and backward."""
    eb = 4 if dtype == "f32" else 2
    B = 4
    rs = (2 * GIB + 4096) // eb
    total = (B - 1) * rs + N
    _need(total * eb)
    assert 2 * rs * eb > 4 * GIB
    x = wl.random_rows(B, N, dtype, seed=N + eb, scale=6.0)
    buf = torch.empty(total, dtype=_tdt(dtype), device="cuda")
    host = torch_view(x, dtype)
    for b in range(B):
        buf[b * rs:b * rs + N] = host[b].cuda()
    xv = buf.as_strided((B, N), (rs, 1))
    want = oracle.lse(x, dtype)
    plans = [None, {"path": "cta", "threads": 512}, {"path": "split", "splits": 3}]
    if N == 64:
        plans.append({"path": "subwarp"})
    for plan in plans:
        got, p = L.lse_forward_plan(xv, plan=plan)
        torch.cuda.synchronize()
        compare(got.cpu().numpy(), want)
    t = np.array([0, N - 1, N // 2, -1], dtype=np.int64)
    want_lp, want_lse = oracle.token_logprob(x, t, dtype)
    lp = L.lse_token_logprob(xv, torch.from_numpy(t).cuda())
    torch.cuda.synchronize()
    compare_logprob(lp.cpu().numpy(), want_lp, want_lse)
    got16, _ = L.lse_forward16(xv)
    compare_e16(got16.cpu().numpy(), want, e16_bound(x, dtype, want))
    g = np.array([1.0, -0.5, 2.0, 0.25])
    dx = torch.empty((B, N), dtype=_tdt(dtype), device="cuda")
    lse_d = torch.from_numpy(want.astype(np.float32)).cuda()
    g_d = torch.from_numpy(g.astype(np.float32)).cuda()
    L.lse_backward_ptr(xv.data_ptr(), dtype, B, N, rs, lse_d.data_ptr(), g_d.data_ptr(),
                       dx.data_ptr(), N)
    torch.cuda.synchronize()
    raw = dx.cpu()
    raw = raw.numpy() if dtype == "f32" else raw.view(torch.int16).numpy().view(np.uint16)
    dec = lambda a: oracle.decode(a, dtype).reshape(a.shape)  # noqa: E731
    compare_backward(dec(raw), dec(x), dtype, want, g, oracle.backward(x, want, g, dtype))
    del buf, xv, dx
    _release()


def test_row_longer_than_2pow31_elements():
    """One bf16 row of 2^31 + 2^20 + 7 elements (4.3 GB): the automatic split
    plan, a target past 2^31, the 16-bit exponentials and a sampled backward."""
    M, k, r = 1 << 20, 2049, 7
    N = k * M + r
    assert N > (1 << 31)
    _need(2 * 2 * N)
    block = wl.random_rows(1, M, "bf16", seed=2031, scale=4.0)
    bt = torch_view(block, "bf16").cuda()
    x = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    x[:k * M].view(k, M).copy_(bt.expand(k, M))
    x[k * M:] = bt[0, :r]
    xv = x.view(1, N)
    l_block = oracle.lse(block, "bf16")[0]
    l_rem = oracle.lse(block[:, :r], "bf16")[0]
    want = float(np.logaddexp(l_block + np.log(k), l_rem))
    got, p = L.lse_forward_plan(xv)
    torch.cuda.synchronize()
    assert p.as_dict()["path"] == "split"
    compare(got.cpu().numpy(), np.array([want]))

    xb = oracle.decode(block, "bf16")
    for t in ((1 << 31) + 12345, N - 1, 0):
        lp = L.lse_token_logprob(xv, torch.tensor([t], device="cuda"))
        torch.cuda.synchronize()
        want_lp = xb[t % M] - want
        compare_logprob(lp.cpu().numpy(), np.array([want_lp]), np.array([want]))

    got16, _ = L.lse_forward16(xv)
    m = np.array([xb.max()])
    e = k * e16_error_sum(block, "bf16", np.array([want]), row_max=m)[0] + \
        e16_error_sum(np.ascontiguousarray(block[:, :r]), "bf16", np.array([want]), row_max=m)[0]
    bound = -np.log1p(-e) + ATOL + RTOL * abs(want)
    compare_e16(got16.cpu().numpy(), np.array([want]), np.array([bound]))

    g = 0.75
    dx = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    lse_d = torch.tensor([want], dtype=torch.float32, device="cuda")
    g_d = torch.tensor([g], dtype=torch.float32, device="cuda")
    L.lse_backward_ptr(xv.data_ptr(), "bf16", 1, N, N, lse_d.data_ptr(), g_d.data_ptr(),
                       dx.data_ptr(), N)
    torch.cuda.synchronize()
    rng = np.random.default_rng(31)
    idx = np.unique(np.concatenate([
        rng.integers(0, N, 4096),
        [0, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, k * M - 1, k * M, N - 1]])).astype(np.int64)
    sample = dx[torch.from_numpy(idx).cuda()].cpu().view(torch.int16).numpy().view(np.uint16)
    want_dx_block = oracle.backward(block, np.array([want]), np.array([g]), "bf16").reshape(-1)
    compare_backward(oracle.decode(sample, "bf16")[None, :], xb[idx % M][None, :], "bf16",
                     np.array([want]), np.array([g]), want_dx_block[idx % M][None, :])
    del x, xv, dx, bt
    _release()


@pytest.mark.parametrize("layout", ["rows_apart", "batches_apart"])
def test_column_strides_beyond_4gib(layout):
    """The value over a non-last dimension with the reduced rows ~2 GiB apart
    (stride_r), or the batch index a ~2 GiB apart (stride_a)."""
    C = 1024
    far = (2 * GIB + 4096) // 4
    if layout == "rows_apart":
        A, R, sa, sr = 1, 4, 4 * far, far
    else:
        A, R, sa, sr = 3, 5, far, C
    total = (A - 1) * sa + (R - 1) * sr + C
    _need(total * 4)
    x = wl.random_rows(A * R, C, "f32", seed=A + R, scale=5.0).reshape(A, R, C)
    buf = torch.empty(total, dtype=torch.float32, device="cuda")
    for a in range(A):
        for rr in range(R):
            buf[a * sa + rr * sr:a * sa + rr * sr + C] = torch.from_numpy(x[a, rr]).cuda()
    want = oracle.lse_strided(np.ascontiguousarray(x).reshape(-1), "f32", A, R, C, R * C, C)
    out = torch.empty(A * C, device="cuda")
    for plan in (None, {"path": "columns_warp"}, {"path": "columns_cta", "lanes_per_row": 2},
                 {"path": "columns_warp", "splits": 2}):
        L.lse_forward_strided_ptr(buf.data_ptr(), "f32", A, R, C, sa, sr, out.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream, plan)
        torch.cuda.synchronize()
        compare(out.cpu().numpy().reshape(A, C), want)
    del buf
    _release()
