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


def test_rotation_copies():
    L2 = bench.L2_BYTES
    assert bench.rotation_copies(262_668_288) == 2          # 2 x 263 MB >= 3 x L2
    assert bench.rotation_copies(1_073_741_824) == 1        # one copy is already 8x L2
    assert bench.rotation_copies(1 << 20) * (1 << 20) >= 3 * L2   # small inputs: many copies
    assert bench.rotation_copies(1 << 20, max_bytes=64 << 20) == 64  # within the memory cap
    assert bench.rotation_copies(0) == 1


def test_block_bounds_and_stats():
    assert bench.block_bounds(200, 4) == [0, 50, 100, 150, 200]
    assert bench.block_bounds(3, 4) == [0, 1, 2, 3]
    assert bench.block_bounds(10, 1) == [0, 10]
    b = bench.block_bounds(30, 3)
    s = bench.block_stats(b, [0.5, 0.4, 0.4])  # ms per block of 10 steps
    assert s["steps"] == 30 and s["blocks"] == 3
    assert abs(s["us_median"] - 40.0) < 1e-9 and abs(s["us_mean"] - 1300 / 30) < 1e-9
    assert abs(s["us_mean_first_half"] - 50.0) < 1e-9          # the first block
    assert abs(s["us_mean_second_half"] - 40.0) < 1e-9         # the last two
    assert bench.block_stats([0], []) == {}
    one = bench.block_stats([0, 7], [0.07])
    assert one["us_mean_first_half"] == one["us_mean_second_half"] == one["us_median"] == 10.0


def test_main_kernel_names_and_sweep_helpers():
    assert bench.main_kernel_name({"path": "cta"}) == "lse_segment_kernel"
    assert bench.main_kernel_name({"path": "rowtile", "slots_per_lane": 8}) == "lse_rowtile_kernel"
    assert bench.main_kernel_name({"path": "rowtile", "slots_per_lane": 0}) == "lse_rowtile_any_kernel"
    B, N = bench.sweep_shape(128256, 4)
    assert N == 128256 and abs(B * N * 4 - bench.SWEEP_BYTES) < N * 4
    assert bench.sweep_shape(1 << 40, 4) == (1, 1 << 40)
    plan = {"path": "cta", "threads": 512, "splits": 1, "lanes_per_row": 0, "slots_per_lane": 0}
    t = bench.sweep_table([{"dtype": "f32", "N": 128256, "B": 1046, "plan": plan,
                            "us_median": 80.0, "gbs": 6700.0, "frac": 1.007}])
    assert "| f32 | 128256 | 1046 | cta T=512 | 80.00 | 6700 | 1.007 |" in t
    assert sorted(bench.SWEEP_N) == bench.SWEEP_N and bench.SWEEP_N[0] == 16


def test_clock_samples_kept_by_window():
    import datetime
    base = datetime.datetime(2026, 12, 2, 12, 0, 0)

    def line(sec, mhz, thermal="Not Active"):
        ts = (base + datetime.timedelta(seconds=sec)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, {thermal}, Not Active, Not Active"

    c = bench.ClockSampler(0)
    c.lines = [line(0.0, 1000), line(1.0, 2070), line(1.1, 2055, "Active"), line(5.0, 900)]
    t0 = base.timestamp()
    s = c.summary(t0 + 0.9, t0 + 1.2)
    assert s["samples_in_window"] == 2 and s["sm_mhz"] == (2070 + 2055) / 2
    assert s["reasons"] == ["hw_thermal_slowdown"] and s["sm_max_mhz"] == 2070
    everything = c.summary(t0 + 100, t0 + 200)  # nothing inside: every sample
    assert everything["samples_in_window"] == 0 and everything["samples"] == 4
    assert bench.ClockSampler.parse("garbage") is None


def test_columns_sweep_helpers():
    assert bench.columns_sweep_shape(64, 1024, 4) == (256 << 20) // (64 * 1024 * 4)
    assert bench.columns_sweep_shape(4096, 16384, 4) == 1
    assert bench.columns_sweep_shape(1 << 20, 1 << 20, 4) == 0
    plan = {"path": "columns_warp", "lanes_per_row": 1, "vector_bytes": 16, "splits": 1}
    q = {"dtype": "bf16", "R": 8, "C": 64, "A": 262144, "plan": plan, "fwd_us": 50.0,
         "fwd_gbs": 5400.0, "fwd_frac": 0.812, "bwd_us": 80.0, "bwd_gbs": 6800.0, "bwd_frac": 1.02}
    t = bench.columns_sweep_table([q, dict(q, plan=dict(plan, path="columns_cta", lanes_per_row=4,
                                                           splits=9, vector_bytes=1))])
    assert "| bf16 | 8 | 64 | 262144 | warp | 50.00 | 5400 | 0.812 | 80.00 | 6800 | 1.020 |" in t
    assert "| cta WT=4 elem P=9 |" in t
    assert "| short |" in bench.columns_sweep_table([dict(q, plan=dict(plan, path="columns_short",
                                                                        lanes_per_row=0))])
    assert bench.main_kernel_name({"path": "columns_short"}) == "lse_cols_short_kernel"
