"""Seeded randomized parity sweep: random dtype, shape, layout, special values
and mapping for every op, each checked against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import compare, compare_logprob, device_rows, torch_view

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402

DTYPES = ["f32", "bf16", "f16"]
SPECIAL = {"f32": (np.nan, np.inf, -np.inf), "bf16": (0x7FC0, 0x7F80, 0xFF80),
           "f16": (0x7E00, 0x7C00, 0xFC00)}


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _random_rows(rng, B, N, dtype):
    scale = float(rng.choice([0.5, 4.0, 30.0]))
    shift = float(rng.choice([0.0, -50.0, 300.0]))
    if dtype == "f16":
        shift = min(shift, 100.0)
    x = wl.random_rows(B, N, dtype, seed=int(rng.integers(1 << 30)), scale=scale, shift=shift)
    if B and N:
        xi = x.view(np.uint16) if dtype != "f32" else x
        for _ in range(int(rng.integers(0, 4))):  # sprinkle special values
            b, n = int(rng.integers(B)), int(rng.integers(N))
            xi[b, n] = SPECIAL[dtype][int(rng.integers(3))]
        if rng.random() < 0.2:
            xi[int(rng.integers(B))] = SPECIAL[dtype][2]  # a whole -inf row
    return x


def _random_plan(rng, N, dtype, aligned, rs):
    """A random plan: vector slots (rows off a 16-byte boundary peel a head and
    a tail slot) or, one time in four, element slots."""
    eb = 4 if dtype == "f32" else 2
    vb = 1 if rng.random() < 0.25 else 16
    epv = 16 // eb if vb == 16 else 1
    slots = N // epv
    nvt = -(-N // epv) if aligned or vb == 1 else N // epv + 2
    choices = [None]
    if N > 0:
        if nvt <= 128:
            G = int(2 ** rng.integers(0, 6))
            if -(-nvt // G) <= 4 or (vb == 16 and G >= 4 and -(-nvt // G) <= 8):
                choices.append({"path": "subwarp", "lanes_per_row": G, "vector_bytes": vb})
        elif nvt <= 256:
            choices.append({"path": "subwarp", "lanes_per_row": 32, "vector_bytes": vb})
        if slots >= 1:
            choices.append({"path": "cta", "threads": int(32 * 2 ** rng.integers(0, 5)),
                            "vector_bytes": vb})
        if slots >= 2:
            choices.append({"path": "split", "splits": int(rng.integers(2, min(slots, 50) + 1)),
                            "threads": int(32 * 2 ** rng.integers(0, 5)), "vector_bytes": vb})
        if aligned and rs == N and N * eb % 16 == 0 and 16 <= N * eb <= 128:
            choices.append({"path": "rowtile"})
    return choices[int(rng.integers(len(choices)))]


@pytest.mark.parametrize("seed", range(150))
def test_random_forward_and_logprob(seed):
    _need_gpu()
    rng = np.random.default_rng(seed)
    dtype = DTYPES[seed % 3]
    B = int(rng.integers(0, 300))
    N = int(np.exp(rng.uniform(0, np.log(40000)))) - 1
    rs = N + int(rng.choice([0, 0, 1, 8, 13]))
    off = int(rng.choice([0, 0, 0, 1, 3]))
    x = _random_rows(rng, B, N, dtype)
    _, xv = device_rows(x, dtype, row_stride=rs, offset=off)
    eb = 4 if dtype == "f32" else 2
    aligned = xv.data_ptr() % 16 == 0 and (rs * eb) % 16 == 0
    plan = _random_plan(rng, N, dtype, aligned, rs)
    want = oracle.lse(x, dtype)
    out = torch.full((B + 4,), float("nan"), device="cuda")
    try:
        got, p = L.lse_forward_plan(xv, plan=plan, out=out[:B])
    except L.LseError:
        if plan and plan.get("path") == "rowtile":
            pytest.skip("rowtile not valid for this layout")
        raise
    torch.cuda.synchronize()
    assert np.all(np.isnan(out[B:].cpu().numpy()))
    compare(got.cpu().numpy(), want)
    t = rng.integers(-2, N + 2, B).astype(np.int64)
    want_lp, want_lse = oracle.token_logprob(x, t, dtype)
    lp, p2 = L.lse_token_logprob(xv, torch.from_numpy(t).cuda(), plan=plan, return_plan=True)
    torch.cuda.synchronize()
    compare_logprob(lp.cpu().numpy(), want_lp, want_lse)


@pytest.mark.parametrize("seed", range(60))
def test_random_strided(seed):
    _need_gpu()
    rng = np.random.default_rng(1000 + seed)
    dtype = DTYPES[seed % 3]
    A, R, C = int(rng.integers(1, 20)), int(rng.integers(1, 700)), int(rng.integers(1, 700))
    x = _random_rows(rng, A * R, C, dtype).reshape(A, R, C)
    pad_c = int(rng.choice([0, 0, 3, 8]))
    sr = C + pad_c
    sa = R * sr + int(rng.choice([0, 8, 5]))
    flat = np.full(A * sa + 16, np.nan if dtype == "f32" else SPECIAL[dtype][0],
                   dtype=np.float32 if dtype == "f32" else np.uint16)
    for a in range(A):
        flat[a * sa:a * sa + R * sr].reshape(R, sr)[:, :C] = x[a] if dtype == "f32" \
            else x[a].view(np.uint16)
    want = oracle.lse_strided(flat, dtype, A, R, C, sa, sr)
    buf = torch_view(flat, dtype).cuda()
    out = torch.empty(A * C, device="cuda")
    plan = [None, {"path": "columns_warp"}, {"path": "columns_cta", "lanes_per_row": 2},
            {"path": "columns_warp", "splits": 2}, {"path": "columns_cta", "splits": 3},
            {"path": "columns_cta", "lanes_per_row": 4, "splits": 2}][seed % 6]
    if plan and plan.get("splits", 0) > R:
        plan = None
    L.lse_forward_strided_ptr(buf.data_ptr(), dtype, A, R, C, sa, sr, out.data_ptr(),
                              torch.cuda.current_stream().cuda_stream, plan)
    torch.cuda.synchronize()
    compare(out.cpu().numpy().reshape(A, C), want)
