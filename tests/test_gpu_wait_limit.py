"""The give-up path of the bulk-copy ring's bounded waits, run on purpose.

lse_set_wait_limit(0) makes every stage wait of LSE_PATH_ROWTILE give up at
its first poll.  Each warp (vector ring) or CTA (any-width ring) then stops,
waits with the default limit for the bulk copies it had already issued, counts
one timeout and exits: the launch returns, lse_wait_timeouts rises, and the
entry point itself returned LSE_OK.  With the default limit restored, the next
call on the same rows is correct.  Nothing here waits on a flag that nothing
sets: every copy that is waited for was issued and lands.
"""
import numpy as np
import pytest

import oracle
from log_sum_exp_gb300 import workloads as wl
from lse_testutil import compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("N,lanes", [(32, None), (8, None), (7, None), (300, None)])
def test_stage_wait_gives_up_then_recovers(N, lanes):
    """N = 32 / 8: the vector ring (128- and 32-byte rows); N = 7: the
    any-width ring, one thread per row; N = 300: the any-width ring with a
    group of lanes per row."""
    _need_gpu()
    B = 40000
    x = wl.generate("short_1048576x32_f32", B=B, N=N) if N == 32 else \
        wl.random_rows(B, N, "f32", seed=N, scale=6.0)
    xd = torch.from_numpy(x).cuda()
    want = oracle.lse(x)
    plan = {"path": "rowtile"}
    if lanes:
        plan["lanes_per_row"] = lanes
    before = L.lse_wait_timeouts()
    out = torch.full((B,), 7.0, device="cuda")
    try:
        L.lse_set_wait_limit(0)
        _, p = L.lse_forward_plan(xd, plan=plan, out=out)  # returns LSE_OK
        torch.cuda.synchronize()  # the launch finishes: nothing hangs
    finally:
        L.lse_set_wait_limit(L.DEFAULT_WAIT_POLLS)
    assert p.as_dict()["path"] == "rowtile"
    after = L.lse_wait_timeouts()
    assert after > before
    # Rows of the stopped warps are left as they were.
    assert np.any(out.cpu().numpy() == 7.0)
    got, p2 = L.lse_forward_plan(xd, plan=plan)
    torch.cuda.synchronize()
    compare(got.cpu().numpy(), want)
    assert L.lse_wait_timeouts() == after
