"""GPU parity of the fused token log-probability (lse_token_logprob) against
the fp64 oracle: logprob[b] = x[b, target[b]] - lse[b]."""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import compare, compare_logprob, device_rows, torch_view

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _targets(B, N, seed, specials=True):
    rng = np.random.default_rng(seed)
    t = rng.integers(0, max(N, 1), B).astype(np.int64)
    if specials and B >= 6:
        t[0], t[1], t[2] = 0, N - 1, -1
        t[3], t[4] = N, 1 << 40
    return t


def run_logprob(xv, target, plan=None, with_lse=True):
    B = xv.shape[0]
    td = torch.from_numpy(target).cuda()
    lse_buf = torch.full((B + 8,), float("nan"), device=xv.device) if with_lse else None
    lp, p = L.lse_token_logprob(xv, td, lse_out=lse_buf[:B] if with_lse else None, plan=plan,
                                return_plan=True)
    torch.cuda.synchronize()
    if with_lse:
        assert np.all(np.isnan(lse_buf[B:].cpu().numpy())), "write past lse_out[B-1]"
    return lp.cpu().numpy(), (lse_buf[:B].cpu().numpy() if with_lse else None), p


@pytest.mark.parametrize("key,B,N", [
    ("vocab_512x128256_f32", None, None),
    ("vocab_8192x32000_bf16", None, None),
    ("short_1048576x32_f32", None, None),
    ("particles_16x16777216_f32", 4, 1 << 22),
    ("small_64x4096_f32", None, None),
])
def test_workload_logprob(key, B, N):
    _need_gpu()
    w = wl.WORKLOADS[key]
    x = wl.generate(key, B=B, N=N)
    Bx, Nx = x.shape
    t = _targets(Bx, Nx, seed=w.index)
    want_lp, want_lse = oracle.token_logprob(x, t, w.dtype)
    xd = torch_view(x, w.dtype).cuda()
    lp, lse, p = run_logprob(xd, t)
    compare(lse, want_lse)
    s = compare_logprob(lp, want_lp, want_lse)
    print(key, p.as_dict()["path"], s)


PLANS = [None, {"path": "cta", "threads": 32}, {"path": "cta", "threads": 512},
         {"path": "split", "splits": 3, "threads": 128}, {"path": "split", "splits": 7, "threads": 256}]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 9, 31, 33, 127, 129, 200, 1000, 1024, 2047, 4097,
                               20001])
def test_logprob_edge_shapes(dtype, N):
    _need_gpu()
    B = 9
    x = wl.random_rows(B, N, dtype, seed=100 + N, scale=5.0)
    if N >= 4:
        xi = x.view(np.uint16) if dtype != "f32" else x
        nan = {"f32": np.nan, "bf16": 0x7FC0, "f16": 0x7E00}[dtype]
        ninf = {"f32": -np.inf, "bf16": 0xFF80, "f16": 0xFC00}[dtype]
        pinf = {"f32": np.inf, "bf16": 0x7F80, "f16": 0x7C00}[dtype]
        xi[5, N // 2] = nan
        xi[6, :] = ninf
        xi[7, 1] = pinf
        xi[8, 2] = ninf
    t = _targets(B, N, seed=N)
    t[8] = 2 if N > 2 else 0  # target a -inf entry
    want_lp, want_lse = oracle.token_logprob(x, t, dtype)
    eb = 4 if dtype == "f32" else 2
    for row_stride, offset in ((N, 0), (N + 5, 1), (N + 8, 0)):
        _, xv = device_rows(x, dtype, row_stride=row_stride, offset=offset)
        # Vector slots on every layout: rows off a 16-byte boundary peel a head
        # and a tail slot; the element mappings are forced on those too.
        aligned = (xv.data_ptr() % 16 == 0) and (row_stride * eb) % 16 == 0
        epv = 16 // eb
        slots = N // epv
        nvt = -(-N // epv) if aligned else N // epv + 2
        plans = list(PLANS)
        if nvt <= 128:
            plans += [{"path": "subwarp", "lanes_per_row": G} for G in (1, 2, 4, 8, 16, 32)
                      if -(-nvt // G) <= 4]
        elif nvt <= 256:
            plans.append({"path": "subwarp", "lanes_per_row": 32})
        plans += [{"path": "subwarp", "lanes_per_row": G} for G in (4, 8, 16)
                  if 4 < -(-nvt // G) <= 8]  # 8 vectors per lane
        if aligned and row_stride == N and N * eb % 16 == 0 and 16 <= N * eb <= 128:
            plans.append({"path": "rowtile"})
        if not aligned:
            plans += [{"path": "cta", "threads": 128, "vector_bytes": 1},
                      {"path": "split", "splits": 3, "threads": 64, "vector_bytes": 1}]
            if N <= 128:
                plans.append({"path": "subwarp", "lanes_per_row": 32, "vector_bytes": 1})
        for plan in plans:
            if plan and plan.get("path") == "split" and \
                    (N if plan.get("vector_bytes") == 1 else slots) < plan["splits"]:
                continue
            for with_lse in (True, False):
                lp, lse, p = run_logprob(xv, t, plan, with_lse)
                try:
                    compare_logprob(lp, want_lp, want_lse)
                    if with_lse:
                        compare(lse, want_lse)
                except AssertionError as e:
                    raise AssertionError(f"stride={row_stride} offset={offset} plan={plan} "
                                         f"ran={p.as_dict()}: {e}") from None


def test_logprob_rowtile_ragged_chunks_and_dtypes():
    """The bulk-copy mapping's epilogue: row counts leaving a partial last
    chunk, every row size and dtype, targets in and out of range."""
    _need_gpu()
    for dtype, eb in (("f32", 4), ("bf16", 2), ("f16", 2)):
        for rb in range(16, 129, 16):
            N = rb // eb
            for B in (1, 255, 2049, 100003):
                x = wl.random_rows(B, N, dtype, seed=3 * B + rb, scale=8.0)
                t = _targets(B, N, seed=B + rb)
                want_lp, want_lse = oracle.token_logprob(x, t, dtype)
                for with_lse in (True, False):
                    lp, lse, p = run_logprob(torch_view(x, dtype).cuda(), t, {"path": "rowtile"},
                                             with_lse)
                    assert p.as_dict()["path"] == "rowtile"
                    compare_logprob(lp, want_lp, want_lse)
                    if with_lse:
                        compare(lse, want_lse)


def test_logprob_empty_rows():
    _need_gpu()
    x = torch.empty((5, 0), device="cuda")
    t = np.zeros(5, np.int64)
    lp, lse, p = run_logprob(x, t)
    assert p.as_dict()["path"] == "empty"
    assert np.all(np.isnan(lp)) and np.all(lse == -np.inf)


def test_logprob_rejects_bad_pointers():
    _need_gpu()
    x = torch.zeros((4, 8), device="cuda")
    lp = torch.empty(4, device="cuda")
    t = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(L.LseError):
        L.lse_token_logprob_ptr(x.data_ptr(), "f32", 4, 8, 8, 0, lp.data_ptr())
    with pytest.raises(L.LseError):
        L.lse_token_logprob_ptr(x.data_ptr(), "f32", 4, 8, 8, t.data_ptr() + 4, lp.data_ptr())
    with pytest.raises(L.LseError):
        L.lse_token_logprob_ptr(x.data_ptr(), "f32", 4, 8, 8, t.data_ptr(), lp.data_ptr() + 2)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_logprob_any_width_ring(dtype):
    """The bulk-copy ring for back-to-back rows of any width with the token
    log-probability epilogue: a thread per row up to 128 bytes plus one
    element, 4-32 lanes per row up to 4 KB; targets in and out of range, on special values, partial
    last chunks and the rows after the last copy, with and without lse_out."""
    _need_gpu()
    eb = 4 if dtype == "f32" else 2
    widths = (1, 3, 5, 7, 9, 31, 33, 129, 257, 1023) if dtype == "f32" else \
        (1, 3, 7, 9, 63, 65, 257, 1025, 2047)
    for N in widths:
        for B in (1, 9, 1001, 20003):
            x = wl.random_rows(B, N, dtype, seed=B + 3 * N, scale=6.0)
            if B >= 9 and N >= 3:
                xi = x.view(np.uint16) if dtype != "f32" else x
                ninf = {"f32": -np.inf, "bf16": 0xFF80, "f16": 0xFC00}[dtype]
                pinf = {"f32": np.inf, "bf16": 0x7F80, "f16": 0x7C00}[dtype]
                nan = {"f32": np.nan, "bf16": 0x7FC0, "f16": 0x7E00}[dtype]
                xi[5, 1] = nan
                xi[6, N - 1] = pinf
                xi[7, :] = ninf
                xi[8, 2] = ninf
            t = _targets(B, N, seed=N * 7 + B)
            if B >= 9:
                t[8] = 2 if N > 2 else 0  # a -inf entry
            want_lp, want_lse = oracle.token_logprob(x, t, dtype)
            xd = torch_view(x, dtype).cuda()
            plans = [{"path": "rowtile"}]
            if N * eb > 128 + eb:  # past a thread per row
                plans += [{"path": "rowtile", "lanes_per_row": G} for G in (4, 32)]
            for plan in plans:
                for with_lse in (True, False):
                    lp, lse, p = run_logprob(xd, t, plan, with_lse)
                    d = p.as_dict()
                    assert d["path"] == "rowtile", d
                    try:
                        compare_logprob(lp, want_lp, want_lse)
                        if with_lse:
                            compare(lse, want_lse)
                    except AssertionError as e:
                        raise AssertionError(f"N={N} B={B} plan={d} lse={with_lse}: {e}") from None
    assert L.lse_wait_timeouts() == 0
