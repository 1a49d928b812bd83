"""GPU parity: liblse (through its C ABI) against the fp64 oracle.

Every finite output must satisfy |gpu - oracle| <= 1e-5 + 1e-6 |oracle|; NaN
and +-inf must match exactly.  Inputs come from the seeded generators and are
handed unchanged to both sides.
"""
import math

import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import compare, compare_e16, compare_logprob, device_rows, e16_bound, torch_view

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run(x_view, plan=None, canary=16):
    """Run lse_forward_plan into a NaN-canaried output buffer; return (out, plan)."""
    B = x_view.shape[0]
    out_buf = torch.full((B + canary,), float("nan"), dtype=torch.float32, device=x_view.device)
    out, p = L.lse_forward_plan(x_view, plan=plan, out=out_buf[:B])
    torch.cuda.synchronize()
    tail = out_buf[B:].cpu().numpy()
    assert np.all(np.isnan(tail)), "write past out[B-1]"
    return out.cpu().numpy(), p


# ---------------------------------------------------------------------------
# The five workloads at full size, automatic plan.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("key", wl.ORDER)
def test_workload_full_size(key):
    _need_gpu()
    w = wl.WORKLOADS[key]
    x = wl.generate(key)
    want = oracle.lse(x, w.dtype)
    xd = torch_view(x, w.dtype).cuda()
    got, p = run(xd)
    s = compare(got, want)
    print(key, p.as_dict(), s)
    del xd
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Edge shapes x dtypes x layouts x every mapping.
# ---------------------------------------------------------------------------
LENGTHS = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255,
           256, 257, 511, 512, 513, 1023, 1024, 1025, 2047, 2048, 2049, 4095, 4096, 4097,
           8191, 12345, 65537, 131073]


def plans_for(N, dtype, vec, aligned=True):
    """Forced plans for rows of N elements.  vec: 16-byte vector slots; rows
    that are not 16-byte aligned (aligned=False) peel a head and a tail slot."""
    eb = 4 if dtype == "f32" else 2
    epv = 16 // eb if vec else 1
    nvt = -(-N // epv) if aligned or not vec else N // epv + 2
    slots = N // epv if vec else N
    plans = [None]
    vb = 16 if vec else 1
    if nvt <= 128:
        G = 1
        while G <= 32:
            if -(-nvt // G) <= 4:
                plans.append({"path": "subwarp", "lanes_per_row": G, "vector_bytes": vb})
            G *= 2
    if 4 < -(-nvt // 32) <= 8:  # a whole warp per row, up to 8 slots per lane
        plans.append({"path": "subwarp", "lanes_per_row": 32, "vector_bytes": vb})
    if vec:  # 4-16 lanes per row with 8 vectors each
        for G in (4, 8, 16):
            if 4 < -(-nvt // G) <= 8:
                plans.append({"path": "subwarp", "lanes_per_row": G, "vector_bytes": vb})
    if slots >= 1:
        for T in (32, 64, 128, 256, 512):
            plans.append({"path": "cta", "threads": T, "vector_bytes": vb})
    for P, T in ((2, 256), (3, 32), (5, 512), (7, 128), (64, 64)):
        if slots >= P:
            plans.append({"path": "split", "splits": P, "threads": T, "vector_bytes": vb})
    return plans


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", LENGTHS)
def test_edge_shapes(dtype, N):
    _need_gpu()
    B = 5
    x = wl.random_rows(B, N, dtype, seed=N, scale=6.0, shift=-2.0)
    # A special value in some rows at the first / last / middle position.
    if N >= 3:
        xi = x.view(np.uint16) if dtype != "f32" else x
        ninf = {"f32": -np.inf, "bf16": 0xFF80, "f16": 0xFC00}[dtype]
        pinf = {"f32": np.inf, "bf16": 0x7F80, "f16": 0x7C00}[dtype]
        nan = {"f32": np.nan, "bf16": 0x7FC0, "f16": 0x7E00}[dtype]
        xi[1, N - 1] = nan
        xi[2, 0] = pinf
        xi[3, :] = ninf
        xi[4, N // 2] = ninf
    want = oracle.lse(x, dtype)
    eb = 4 if dtype == "f32" else 2
    layouts = [(N, 0), (N + 8, 0), (N + 1, 0), (N, 1)]
    for row_stride, offset in layouts:
        buf, xv = device_rows(x, dtype, row_stride=row_stride, offset=offset)
        aligned = (xv.data_ptr() % 16 == 0) and (row_stride * eb) % 16 == 0
        plans = plans_for(N, dtype, aligned)
        if not aligned:  # the vector mappings with the head and tail peeled
            plans += plans_for(N, dtype, True, aligned=False)[1:]
        if row_stride == N and N * eb <= 128 and xv.data_ptr() % 16 == 0:
            plans.append({"path": "rowtile"})  # vector ring, or element reads for other widths
        for plan in plans:
            got, p = run(xv, plan)
            try:
                compare(got, want)
            except AssertionError as e:
                raise AssertionError(f"layout stride={row_stride} offset={offset} "
                                     f"plan={plan} ran={p.as_dict()}: {e}") from None


def test_scalar_path_forced_on_aligned_rows():
    _need_gpu()
    for dtype in ("f32", "bf16", "f16"):
        x = wl.random_rows(9, 3001, dtype, seed=3)
        want = oracle.lse(x, dtype)
        _, xv = device_rows(x, dtype)
        for plan in ({"vector_bytes": 1}, {"path": "split", "splits": 4, "vector_bytes": 1}):
            got, p = run(xv, plan)
            assert p.vector_bytes == 1
            compare(got, want)


# ---------------------------------------------------------------------------
# Degenerate sizes and special values.
# ---------------------------------------------------------------------------
def test_empty_rows_give_neg_inf():
    _need_gpu()
    for dtype in ("f32", "bf16", "f16"):
        x = np.zeros((7, 0), dtype=np.float32 if dtype == "f32" else np.uint16)
        _, xv = device_rows(x, dtype)
        got, p = run(xv)
        assert p.as_dict()["path"] == "empty"
        assert np.all(got == -np.inf)


def test_zero_rows_is_noop():
    _need_gpu()
    x = torch.empty((0, 100), device="cuda")
    out = L.lse_forward(x)
    assert out.shape == (0,)


def test_single_element_rows_exact():
    """N = 1: the result is the element itself (every bf16 / f16 bit pattern)."""
    _need_gpu()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(-1, 1)
    for dtype in ("bf16", "f16"):
        want = oracle.lse(bits, dtype)
        got, _ = run(torch_view(bits, dtype).cuda())
        compare(got, want, atol=0.0, rtol=0.0)


def test_extreme_magnitudes():
    _need_gpu()
    big = np.float32(3.0e38)
    rows = [
        [big, big], [-big, big], [big, -np.inf], [-big, -big],
        [1e-40, -1e-40], [0.0, -0.0], [-1e30, -1e30 + 1e24], [88.7, 88.7, 88.7],
        [-103.0, -103.0], [np.inf, -np.inf], [np.nan, -np.inf], [-np.inf, np.nan],
    ]
    n = max(len(r) for r in rows)
    x = np.full((len(rows), n), -np.inf, dtype=np.float32)
    for i, r in enumerate(rows):
        x[i, :len(r)] = r
    want = oracle.lse(x)
    for plan in (None, {"path": "cta", "threads": 32}, {"path": "cta", "threads": 256},
                 {"path": "cta", "threads": 512}):
        got, _ = run(torch.from_numpy(x).cuda(), plan)
        compare(got, want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_magnitudes_every_mapping(dtype):
    """Rows of 32 elements whose maximum is far beyond 2^24 (the shift's
    rounding residual in the one-FFMA term form would then be large: 6e21 at
    -1e30) or near the top of the range, beside ordinary rows, on every
    mapping that takes such rows: sub-warp groups, the bulk-copy ring,
    CTA and split."""
    _need_gpu()
    N = 32
    rng = np.random.default_rng(9)
    base = rng.normal(0, 3, (16, N)).astype(np.float32)
    centres = [-1e30, 1e30, 3e9, -3e9, 2.0 ** 24 + 1.0, -7e7, 3e38, -3e38, 1e20, 0.0,
               5e4, -5e4, 2.0 ** 127, 1e36, -1e36, 1.5e19]
    x = np.zeros_like(base)
    for i, c in enumerate(centres):
        spread = abs(c) * 1e-6 if c else 1.0
        x[i] = np.float32(c) + (base[i] * spread).astype(np.float32)
    x[6, 5] = np.float32(3.4e38)
    if dtype == "bf16":
        x = wl.f32_to_bf16_bits(x)
    want = oracle.lse(x, dtype)
    xd = torch_view(x, dtype).cuda()
    eb = 4 if dtype == "f32" else 2
    plans = [None, {"path": "subwarp", "lanes_per_row": 2}, {"path": "subwarp", "lanes_per_row": 8},
             {"path": "subwarp", "lanes_per_row": 32}, {"path": "cta", "threads": 64},
             {"path": "split", "splits": 2}]
    if N * eb <= 128:
        plans.append({"path": "rowtile"})
    for plan in plans:
        got, p = run(xd, plan)
        try:
            compare(got, want)
        except AssertionError as e:
            raise AssertionError(f"plan {p.as_dict()}: {e}") from None
    lp = L.lse_token_logprob(xd, torch.zeros(16, dtype=torch.int64, device="cuda"))
    want_lp, want_lse = oracle.token_logprob(x, np.zeros(16, dtype=np.int64), dtype)
    compare_logprob(lp.cpu().numpy(), want_lp, want_lse)


def test_special_value_in_every_split_segment():
    """NaN / +inf / only -inf inside one segment of a split row."""
    _need_gpu()
    N, P = 40000, 8
    base = wl.random_rows(1, N, "f32", seed=21)[0]
    cases = []
    for seg in range(P):
        pos = seg * (N // P) + 17
        for val in (np.nan, np.inf):
            r = base.copy()
            r[pos] = val
            cases.append(r)
    r = np.full(N, -np.inf, np.float32)
    r[N - 1] = 3.0
    cases.append(r)
    x = np.stack(cases)
    want = oracle.lse(x)
    got, p = run(torch.from_numpy(x).cuda(), {"path": "split", "splits": P, "threads": 256})
    assert p.splits == P
    compare(got, want)


def test_deterministic():
    _need_gpu()
    x = torch.from_numpy(wl.generate("vocab_512x128256_f32", B=64)).cuda()
    a = L.lse_forward(x).cpu().numpy()
    for _ in range(3):
        assert np.array_equal(L.lse_forward(x).cpu().numpy(), a)


def test_one_dimensional_input():
    _need_gpu()
    x = wl.random_rows(1, 777, "f32", seed=2)
    got = L.lse_forward(torch.from_numpy(x[0]).cuda())
    assert got.shape == ()
    compare(np.array([got.item()]), oracle.lse(x))


def test_plan_query_matches_forward():
    _need_gpu()
    for key in wl.ORDER:
        w = wl.WORKLOADS[key]
        q = L.lse_plan_query(dtype=w.dtype, B=w.B, N=w.N)
        assert q["launches"] in (1, 2)
        if key.startswith("short"):
            assert q["path"] == "rowtile"
        if key.startswith("particles"):
            assert q["path"] == "split"


def test_invalid_arguments_raise():
    _need_gpu()
    x = torch.zeros((4, 8), device="cuda")
    out = torch.empty(4, device="cuda")
    with pytest.raises(L.LseError) as e:
        L.lse_forward_ptr(x.data_ptr(), "f32", 4, 8, 7, out.data_ptr())
    assert e.value.status == 1
    with pytest.raises(L.LseError):
        L.lse_forward_ptr(x.data_ptr(), "f32", 4, 8, 8, out.data_ptr() + 2)
    with pytest.raises(L.LseError):
        L.lse_forward_plan(x, plan={"path": "subwarp", "lanes_per_row": 3})
    with pytest.raises(L.LseError):
        L.lse_forward_plan(x, plan={"path": "split", "splits": 100})
    assert L.load().lse_forward(x.data_ptr(), 7, 4, 8, 8, out.data_ptr(), None) == 2
    with pytest.raises(ValueError):
        L.lse_forward(x.t())  # last dimension not unit-stride


def test_host_entry_point_pinned_and_pageable():
    """lse_forward_host: pinned buffers are used in place (zero copy), pageable
    ones are staged through device memory; every combination gives the oracle."""
    _need_gpu()
    x = wl.generate("vocab_512x128256_f32", B=32)
    x[3, 5] = np.nan
    x[4, :] = -np.inf
    want = oracle.lse(x)
    B, N = x.shape
    for pin_x in (True, False):
        for pin_out in (True, False):
            xt = torch.from_numpy(x.copy())
            if pin_x:
                xt = xt.pin_memory()
            out = torch.full((B,), 7.0, dtype=torch.float32)
            if pin_out:
                out = out.pin_memory()
            L.lse_forward_host_ptr(xt.data_ptr(), "f32", B, N, N, out.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
            compare(out.numpy(), want)
    # Padded rows through the host entry.
    padded = np.full((B, N + 3), np.nan, dtype=np.float32)
    padded[:, :N] = x
    pt = torch.from_numpy(padded).pin_memory()
    out = torch.empty(B, dtype=torch.float32)
    L.lse_forward_host_ptr(pt.data_ptr(), "f32", B, N, N + 3, out.data_ptr())
    compare(out.numpy(), want)
    compare(L.lse_forward_host(torch.from_numpy(x)).numpy(), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_host_entry_point_dtypes(dtype):
    """lse_forward_host for every element type, page-locked and pageable input."""
    _need_gpu()
    x = wl.random_rows(64, 1000, dtype, seed=17, scale=7.0)
    want = oracle.lse(x, dtype)
    for pin in (True, False):
        xt = torch_view(x.copy(), dtype)
        if pin:
            xt = xt.pin_memory()
        out = torch.full((64,), 7.0, dtype=torch.float32).pin_memory()
        L.lse_forward_host_ptr(xt.data_ptr(), dtype, 64, 1000, 1000, out.data_ptr())
        compare(out.numpy(), want)


def test_host_entry_point_short_rows_bulk_copy():
    """Short back-to-back rows from page-locked host memory take the bulk-copy
    mapping, whose copies then read host memory in place: full short-row
    workload against the oracle, and no bounded wait gave up."""
    _need_gpu()
    x = wl.generate("short_1048576x32_f32")
    B, N = x.shape
    assert L.lse_plan_query(dtype="f32", B=B, N=N, row_stride=N)["path"] == "rowtile"
    before = L.lse_wait_timeouts()
    xt = torch.from_numpy(x).pin_memory()
    out = torch.empty(B, dtype=torch.float32).pin_memory()
    L.lse_forward_host_ptr(xt.data_ptr(), "f32", B, N, N, out.data_ptr())
    compare(out.numpy(), oracle.lse(x))
    assert L.lse_wait_timeouts() == before


def test_cuda_graph_capture_and_replay():
    _need_gpu()
    for key, B in (("small_64x4096_f32", None), ("particles_16x16777216_f32", 2)):
        w = wl.WORKLOADS[key]
        N = w.N if B is None else 1 << 20
        x = wl.generate(key, B=B, N=N)
        xd = torch.from_numpy(x).cuda()
        out = torch.empty(x.shape[0], device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            L.lse_forward(xd, out=out)  # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            L.lse_forward(xd, out=out)
        out.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        compare(out.cpu().numpy(), oracle.lse(x))


def test_tolerance_bar_is_met_with_margin():
    """The worst finite error on the long split rows stays below half the bar."""
    _need_gpu()
    x = wl.generate("particles_16x16777216_f32", B=4)
    s = compare(run(torch.from_numpy(x).cuda())[0], oracle.lse(x))
    assert s["max_err_over_tol"] < 0.5, s
    assert math.isfinite(s["max_abs_err"])


def test_concurrent_streams_split_scratch():
    """Split-row calls on two streams at once: each gets its own stream-ordered
    scratch, so neither disturbs the other."""
    _need_gpu()
    xs = [wl.generate("particles_16x16777216_f32", B=4, N=1 << 21, seed=s) for s in (1, 2)]
    wants = [oracle.lse(x) for x in xs]
    ds = [torch.from_numpy(x).cuda() for x in xs]
    streams = [torch.cuda.Stream() for _ in ds]
    outs = [torch.empty(4, device="cuda") for _ in ds]
    torch.cuda.synchronize()
    for _ in range(20):
        for d, st, o in zip(ds, streams, outs):
            L.lse_forward_plan(d, plan={"path": "split", "splits": 64}, out=o, stream=st)
    torch.cuda.synchronize()
    for o, w in zip(outs, wants):
        compare(o.cpu().numpy(), w)


def test_allocation_failure_is_reported():
    """A staging allocation larger than the device reports LSE_ERR_ALLOC
    (host-side failure: nothing is launched, the host buffer is not read)."""
    _need_gpu()
    small = np.zeros(16, np.float32)
    out = np.zeros(1 << 10, np.float32)
    free, total = torch.cuda.mem_get_info()
    n = int(total // 4 * 2)  # twice the device memory, in f32 elements
    with pytest.raises(L.LseError) as e:
        L.lse_forward_host_ptr(small.ctypes.data, "f32", 1 << 10, n // (1 << 10), n // (1 << 10),
                               out.ctypes.data)
    assert e.value.status == 3
    # The failure is reported once, by status; the runtime is left clean for
    # the caller's next CUDA call.
    torch.ones(3, device="cuda").sum().item()


def test_graph_capture_all_ops():
    """lse_token_logprob, lse_backward, lse_forward_strided, lse_backward_strided
    and lse_forward16 replay correctly from a CUDA graph (split plans included)."""
    _need_gpu()
    x = wl.generate("particles_16x16777216_f32", B=3, N=1 << 20)
    t = np.array([0, 5, (1 << 20) - 1], np.int64)
    xd = torch.from_numpy(x).cuda()
    td = torch.from_numpy(t).cuda()
    lse_d = torch.from_numpy(oracle.lse(x).astype(np.float32)).cuda()
    g_d = torch.ones(3, device="cuda")
    x3 = wl.generate_columns("pcsum_512x64x1024_f32", A=8)
    x3d = torch.from_numpy(x3).cuda()
    lp = torch.empty(3, device="cuda")
    dx = torch.empty_like(xd)
    col = torch.empty(8 * 1024, device="cuda")
    col_lse = torch.from_numpy(oracle.lse_strided(x3.reshape(-1), "f32", 8, 64, 1024, 64 * 1024,
                                                  1024).astype(np.float32)).cuda()
    col_g = torch.ones(8 * 1024, device="cuda")
    dx3 = torch.empty_like(x3d)
    v16 = torch.empty(3, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def ops(stream):
        h = stream.cuda_stream
        L.lse_token_logprob_ptr(xd.data_ptr(), "f32", 3, 1 << 20, 1 << 20, td.data_ptr(),
                                lp.data_ptr(), 0, h, L._binding._as_plan({"path": "split", "splits": 8}))
        L.lse_backward_ptr(xd.data_ptr(), "f32", 3, 1 << 20, 1 << 20, lse_d.data_ptr(),
                           g_d.data_ptr(), dx.data_ptr(), 1 << 20, h)
        L.lse_forward_strided_ptr(x3d.data_ptr(), "f32", 8, 64, 1024, 64 * 1024, 1024,
                                  col.data_ptr(), h, {"path": "columns_warp", "splits": 2})
        L.lse_backward_strided_ptr(x3d.data_ptr(), "f32", 8, 64, 1024, 64 * 1024, 1024,
                                   col_lse.data_ptr(), col_g.data_ptr(), dx3.data_ptr(),
                                   64 * 1024, 1024, h)
        L.lse_forward16_ptr(xd.data_ptr(), "f32", 3, 1 << 20, 1 << 20, v16.data_ptr(), h,
                            L._binding._as_plan({"path": "split", "splits": 8}))

    with torch.cuda.stream(s):
        ops(s)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ops(torch.cuda.current_stream())
    lp.fill_(0)
    dx.fill_(0)
    col.fill_(0)
    dx3.fill_(0)
    v16.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    want_lp, want_lse = oracle.token_logprob(x, t)
    compare(lp.cpu().numpy(), want_lp, scale=np.abs(want_lp) + np.abs(want_lse))
    compare(col.cpu().numpy().reshape(8, 1024),
            oracle.lse_strided(x3.reshape(-1), "f32", 8, 64, 1024, 64 * 1024, 1024))
    assert np.allclose(dx.sum(dim=1).cpu().numpy(), 1.0, rtol=1e-4)
    assert np.allclose(dx3.sum(dim=1).cpu().numpy(), 1.0, rtol=1e-4)
    want = oracle.lse(x)
    assert np.all(np.abs(v16.cpu().numpy() - want) < 3e-3)


def test_rowtile_any_width_ragged():
    """The bulk-copy ring for back-to-back rows whose width is not a multiple of
    16 bytes (element reads from shared memory; the last < 16/gcd(width, 16)
    rows come from global memory), every dtype, odd widths and row counts."""
    _need_gpu()
    for dtype, eb, Ns in (("f32", 4, (1, 2, 3, 5, 6, 7, 9, 13, 17, 31, 33)),
                          ("bf16", 2, (1, 2, 3, 5, 7, 9, 12, 17, 33, 63, 65)),
                          ("f16", 2, (3, 5, 12, 31, 65))):
        for N in Ns:
            for B in (1, 7, 255, 2049, 100003):
                x = wl.random_rows(B, N, dtype, seed=B + 7 * N, scale=8.0)
                got, p = run(torch_view(x, dtype).cuda(), {"path": "rowtile"})
                d = p.as_dict()
                assert d["path"] == "rowtile" and d["slots_per_lane"] == 0, d
                assert d["lanes_per_row"] == 1, d  # a thread per row up to 128 bytes + one element
                compare(got, oracle.lse(x, dtype))
    assert L.lse_wait_timeouts() == 0


def test_thread_rows_past_128_bytes():
    """Rows of 128 bytes plus one element (f32 N = 33, 16-bit N = 65) on the
    thread-per-row ring, whose chunks then hold fewer rows than threads: the
    row value and the token log-probability, special values, ragged row counts,
    forced and (with enough rows) chosen automatically."""
    _need_gpu()
    for dtype, N in (("f32", 33), ("bf16", 65), ("f16", 65)):
        for B in (7, 249, 400003):
            plan = None if B == 400003 else {"path": "rowtile"}  # enough rows to choose it alone
            x = wl.random_rows(B, N, dtype, seed=B + N, scale=6.0, shift=-1.0)
            xi = x.view(np.uint16) if dtype != "f32" else x
            nan, pinf, ninf = {"f32": (np.nan, np.inf, -np.inf), "bf16": (0x7FC0, 0x7F80, 0xFF80),
                               "f16": (0x7E00, 0x7C00, 0xFC00)}[dtype]
            xi[B - 1, N - 1] = nan
            xi[B // 2, 0] = pinf
            xi[B // 3, :] = ninf
            xd = torch_view(x, dtype).cuda()
            got, p = run(xd, plan)
            d = p.as_dict()
            assert d["path"] == "rowtile" and d["lanes_per_row"] == 1 and d["slots_per_lane"] == 0, d
            compare(got, oracle.lse(x, dtype))
            t = np.arange(B, dtype=np.int64) * 5 % (N + 2) - 1
            want_lp, want_lse = oracle.token_logprob(x, t, dtype)
            lp, pl = L.lse_token_logprob(xd, torch.from_numpy(t).cuda(), plan=plan, return_plan=True)
            assert pl.as_dict()["path"] == "rowtile" and pl.as_dict()["lanes_per_row"] == 1
            compare_logprob(lp.cpu().numpy(), want_lp, want_lse)
    assert L.lse_wait_timeouts() == 0


def test_short_row_mapping_rule():
    """Automatic choice between the bulk-copy ring and the sub-warp mapping for
    back-to-back rows of 16..128 bytes (the measured rule): the ring for every
    width but f32 rows of 2 vectors."""
    _need_gpu()
    for dtype, eb in (("f32", 4), ("bf16", 2), ("f16", 2)):
        for nv in range(1, 9):
            N = nv * 16 // eb
            q = L.lse_plan_query(dtype=dtype, B=1 << 20, N=N, row_stride=N)
            ring = not (eb == 4 and nv == 2)
            assert q["path"] == ("rowtile" if ring else "subwarp"), (dtype, nv, q)
            # not back to back, or too few rows: never the ring
            assert L.lse_plan_query(dtype=dtype, B=1 << 20, N=N, row_stride=N + 16 // eb)["path"] \
                == "subwarp"
            assert L.lse_plan_query(dtype=dtype, B=1000, N=N, row_stride=N)["path"] == "subwarp"


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_rowtile_grouped_rows(dtype):
    """The bulk-copy ring for back-to-back rows of 129 bytes to 4 KB (any
    width): groups of 4-32 lanes fold each row from 16-byte reads of the
    staged chunk, masking the neighbouring rows' elements in the row's first
    and last vectors.  Partial last chunks, fewer rows than one alignment
    period, special values, every group size."""
    _need_gpu()
    eb = 4 if dtype == "f32" else 2
    for rb in (130, 134, 144, 252, 516, 1000, 1026, 2048, 2050, 4094, 4096):
        if rb % eb or rb <= 128 + eb:  # up to 128 bytes + one element: a thread per row
            continue
        N = rb // eb
        for B in (1, 3, 9, 1001, 20003):
            x = wl.random_rows(B, N, dtype, seed=B + rb, scale=6.0)
            if B >= 9:
                xi = x.view(np.uint16) if dtype != "f32" else x
                ninf = {"f32": -np.inf, "bf16": 0xFF80, "f16": 0xFC00}[dtype]
                pinf = {"f32": np.inf, "bf16": 0x7F80, "f16": 0x7C00}[dtype]
                nan = {"f32": np.nan, "bf16": 0x7FC0, "f16": 0x7E00}[dtype]
                xi[1, 0] = nan
                xi[2, N - 1] = pinf
                xi[3, :] = ninf
                xi[4, 0] = pinf
                xi[4, N - 1] = nan
            want = oracle.lse(x, dtype)
            xd = torch_view(x, dtype).cuda()
            for G in (None, 4, 8, 16, 32):
                plan = {"path": "rowtile"} if G is None else {"path": "rowtile", "lanes_per_row": G}
                got, p = run(xd, plan)
                d = p.as_dict()
                assert d["path"] == "rowtile" and d["slots_per_lane"] == 0, d
                try:
                    compare(got, want)
                except AssertionError as e:
                    raise AssertionError(f"rb={rb} B={B} plan={d}: {e}") from None
    assert L.lse_wait_timeouts() == 0


def test_any_width_ring_rule():
    """Back-to-back rows of other widths of 32 to 128 bytes take the any-width
    ring, a thread per row, when there are rows for every CTA (row value and
    token log-probability); shorter rows and the 16-bit exponential entry
    point keep the register mappings."""
    _need_gpu()
    for dtype, eb in (("f32", 4), ("bf16", 2), ("f16", 2)):
        for N in (1, 3, 5, 7, 9, 17, 128 // eb - 1):
            # (a query only: 2^26 rows fill every CTA's chunk for any width)
            q = L.lse_plan_query(dtype=dtype, B=1 << 26, N=N, row_stride=N)
            if N * eb < 32:
                assert q["path"] == "subwarp", (dtype, N, q)
                continue
            assert q["path"] == "rowtile" and q["slots_per_lane"] == 0, (dtype, N, q)
            assert L.lse_plan_query(dtype=dtype, B=1000, N=N, row_stride=N)["path"] == "subwarp"
            assert L.lse_plan_query(dtype=dtype, B=1 << 26, N=N, row_stride=N + 1)["path"] \
                == "subwarp"
    # Rows over 512 bytes: the grouped ring where the sub-warp slots would be
    # a quarter empty or more (f32, or 16-bit rows up to 1.5 KB) or cannot hold
    # the row, the sub-warp mapping otherwise.
    for dtype, N, ring, lanes in (("f32", 129, True, 4), ("f32", 520, True, 16),
                                  ("bf16", 1020, False, 0), ("bf16", 2047, True, 16),
                                  ("bf16", 520, True, 4), ("f32", 300, False, 0),
                                  ("f32", 128, False, 0), ("f32", 68, False, 0),
                                  ("f32", 1001, False, 0), ("bf16", 800, False, 0)):
        q = L.lse_plan_query(dtype=dtype, B=1 << 22, N=N, row_stride=N)
        if ring:
            assert q["path"] == "rowtile" and q["lanes_per_row"] == lanes, (dtype, N, q)
        else:
            assert q["path"] == "subwarp", (dtype, N, q)
    x = wl.random_rows(1 << 20, 13, "f32", seed=55, scale=4.0)  # >= 768 rows per CTA
    xd = torch.from_numpy(x).cuda()
    want = oracle.lse(x, "f32")
    got, p = run(xd, None)
    assert p.as_dict()["path"] == "rowtile"
    compare(got, want)
    g16, p16 = L.lse_forward16(xd)
    assert p16.as_dict()["path"] == "subwarp"
    compare_e16(g16.cpu().numpy(), want, e16_bound(x, "f32", want))
    t = np.arange(x.shape[0], dtype=np.int64) % 13
    lp, pl = L.lse_token_logprob(xd, torch.from_numpy(t).cuda(), return_plan=True)
    assert pl.as_dict()["path"] == "rowtile"
    want_lp, want_lse = oracle.token_logprob(x, t, "f32")
    compare_logprob(lp.cpu().numpy(), want_lp, want_lse)
    # The same for rows of 516 bytes (the grouped ring for the row value and
    # the token log-probability).
    x = wl.random_rows(1 << 16, 129, "f32", seed=56, scale=4.0)
    xd = torch.from_numpy(x).cuda()
    want = oracle.lse(x, "f32")
    got, p = run(xd, None)
    assert p.as_dict()["path"] == "rowtile" and p.as_dict()["lanes_per_row"] == 4
    compare(got, want)
    g16, p16 = L.lse_forward16(xd)
    assert p16.as_dict()["path"] == "subwarp"
    compare_e16(g16.cpu().numpy(), want, e16_bound(x, "f32", want))
    t = np.arange(x.shape[0], dtype=np.int64) % 129
    lp, pl = L.lse_token_logprob(xd, torch.from_numpy(t).cuda(), return_plan=True)
    assert pl.as_dict()["path"] == "rowtile"
    want_lp, want_lse = oracle.token_logprob(x, t, "f32")
    compare_logprob(lp.cpu().numpy(), want_lp, want_lse)


def test_short_rows_both_mappings_full_size():
    """The 1048576 x 32 workload through the bulk-copy ring (default) and the
    register sub-warp kernel (forced)."""
    _need_gpu()
    x = wl.generate("short_1048576x32_f32")
    want = oracle.lse(x)
    xd = torch.from_numpy(x).cuda()
    for plan in (None, {"path": "rowtile"}, {"path": "subwarp"}):
        got, p = run(xd, plan)
        if plan is None:
            assert p.as_dict()["path"] == "rowtile"
        compare(got, want)


def test_rowtile_ragged_chunks_and_dtypes():
    """Row counts that leave a partial last chunk, for every row size and dtype."""
    _need_gpu()
    for dtype, eb in (("f32", 4), ("bf16", 2), ("f16", 2)):
        for rb in range(16, 129, 16):
            N = rb // eb
            for B in (1, 255, 2049, 100003):
                x = wl.random_rows(B, N, dtype, seed=B + rb, scale=8.0)
                got, p = run(torch_view(x, dtype).cuda(), {"path": "rowtile"})
                assert p.as_dict()["path"] == "rowtile"
                compare(got, oracle.lse(x, dtype))


def test_no_wait_timed_out():
    """No bounded device-side wait gave up during the tests above."""
    _need_gpu()
    torch.cuda.synchronize()
    assert L.lse_wait_timeouts() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_subwarp_three_and_six_slots(dtype):
    """The 3- and 6-slot sub-warp variants (rows just past a power of two of
    slots), and the 5- and 7-slot ones of a whole warp per row: the row value,
    the token log-probability and the 16-bit exponentials, on rows that start
    on a 16-byte boundary and on rows that do not (their covering vectors take
    one or two more slots), with special values at the first and the last
    element."""
    _need_gpu()
    eb = 4 if dtype == "f32" else 2
    epv = 16 // eb
    seen = set()
    for nvec, lanes in ((3, 1), (5, 2), (9, 4), (11, 4), (18, 4), (21, 4), (40, 8), (90, 16),
                        (170, 32), (140, 32), (200, 32)):
        for extra, offset in ((0, 0), (1, 0), (0, 1), (epv - 1, 1)):
            N = nvec * epv + extra
            B = 37
            x = wl.random_rows(B, N, dtype, seed=N + offset, scale=6.0, shift=-1.0)
            xi = x.view(np.uint16) if dtype != "f32" else x
            nan, pinf, ninf = {"f32": (np.nan, np.inf, -np.inf), "bf16": (0x7FC0, 0x7F80, 0xFF80),
                               "f16": (0x7E00, 0x7C00, 0xFC00)}[dtype]
            xi[1, 0], xi[2, N - 1], xi[3, :] = nan, pinf, ninf
            xi[4, :] = ninf
            xi[4, N - 1] = 0
            want = oracle.lse(x, dtype)
            _, xv = device_rows(x, dtype, row_stride=N + 5, offset=offset)
            plan = {"path": "subwarp", "lanes_per_row": lanes, "vector_bytes": 16}
            try:
                got, p = run(xv, plan)
            except L.LseError:
                continue  # more slots than this group can hold
            V = p.as_dict()["slots_per_lane"]
            seen.add(V)
            try:
                compare(got, want)
                t = np.arange(B, dtype=np.int64) * 7 % (N + 2) - 1  # includes -1 and N
                want_lp, want_lse = oracle.token_logprob(x, t, dtype)
                lp, pl = L.lse_token_logprob(xv, torch.from_numpy(t).cuda(), plan=plan, return_plan=True)
                assert pl.as_dict()["slots_per_lane"] == V
                compare_logprob(lp.cpu().numpy(), want_lp, want_lse)
                g16, p16 = L.lse_forward16(xv, plan=plan)
                assert p16.as_dict()["slots_per_lane"] == V
                compare_e16(g16.cpu().numpy(), want, e16_bound(x, dtype, want))
            except AssertionError as e:
                raise AssertionError(f"N={N} offset={offset} plan={p.as_dict()}: {e}") from None
    assert {3, 5, 6, 7} <= seen, seen
