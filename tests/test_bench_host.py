"""bench.py host logic on CPU: rank seeds and the max-over-ranks timing with a
world_size-2 gloo process group (no GPU)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
from log_sum_exp_gb300 import workloads as wl  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        bench.barrier()
        got = bench.reduce_max(10.0 + 5.0 * rank)
        seed = bench.rank_seed(wl.WORKLOADS[bench.DEFAULT_WORKLOAD], rank)
        results[rank] = (got, seed)
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_rank_seeds_gloo():
    world = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] != res[1][1]


def test_single_process_helpers():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.dist_env()[1] >= 1
    peak, src = bench.measured_peaks()
    assert peak > 0 and isinstance(src, str)
    assert len(bench.kernel_source_hash()) == 16


def test_reference_arm_bounded_and_complete(capsys, monkeypatch):
    """--impl reference times the oracle on the host: each step is a sample
    sized from this host's measured oracle speed so the whole run stays near
    the budget whatever --steps is; the line carries the contract's keys."""
    import json
    import time

    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 2.0)
    t0 = time.perf_counter()
    bench.main(["--impl", "reference", "--steps", "400", "--warmup", "3"])
    elapsed = time.perf_counter() - t0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert elapsed < 30, elapsed
    assert line["impl"] == "reference" and line["steps"] == 400 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["gpu_launches"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["rows_per_step"] >= 1
