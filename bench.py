"""Benchmark of the row-wise log-sum-exp on GB300: prints ONE JSON line.

A step is one lse_forward call (every kernel of the path) over one batch of
the workload, inputs already in HBM.  ``value`` is the algorithmic HBM bytes
of all ranks' steps (B*N*elem read + B*4 written) divided by the max-over-ranks
time, in GB/s.  The default workload is the paper's profiled shape
(B, N) = (512, 128256) in f32 ("Speeding up Log-Sum-Exp ...", Sec. 2.1, Fig. 1;
Tables 6 and 7 use the same shape).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload KEY]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from log_sum_exp_gb300 import workloads as wl  # noqa: E402

METRIC = "row-wise LSE achieved HBM GB/s (% of GB300 peak) and us/call, 1 GPU"
DEFAULT_WORKLOAD = "vocab_512x128256_f32"
DEFAULT_COLUMNS = "pcsum_512x64x1024_f32"
L2_BYTES = 129 * 10**6
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0  # public HBM3e bandwidth of the part, for a labelled second percentage
EVENT_EVERY = 16
OP_NAMES = {"forward": "row value", "forward16": "row value, reduced-bit exponentials",
            "logprob": "fused token log-probability",
            "backward": "backward dx = g exp(x - lse)", "columns": "value over a non-last dim",
            "columns_backward": "backward of the value over a non-last dim"}
COLUMN_OPS = ("columns", "columns_backward")
KERNEL_SOURCES = ["lse_api.cu", "lse_kernels.cuh", "lse_device.cuh", "lse_internal.h",
                  "lse_kernels_f32.cu", "lse_kernels_bf16.cu", "lse_kernels_f16.cu",
                  "lse_logprob_f32.cu", "lse_logprob_bf16.cu", "lse_logprob_f16.cu",
                  "lse_backward.cu", "lse_strided.cu", "lse_rowtile.cu", "lse_ex16_f32.cu",
                  "lse_ex16_bf16.cu", "lse_ex16_f16.cu"]


# ---------------------------------------------------------------------------
# Host-side helpers (also exercised by the CPU tests).
# ---------------------------------------------------------------------------
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(workload: wl.Workload, rank: int) -> int:
    """Each rank draws its own batch of the same workload (weak scaling)."""
    return workload.seed + 7919 * rank


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None) -> None:
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def kernel_source_hash(files: list[str] | None = None) -> str:
    """sha256 (16 hex digits) of kernel source files under the package's csrc/."""
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES if files is None else files):
        with open(os.path.join(ROOT, "log_sum_exp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no measured peak file)"


def backward_kernel(N, eb):
    """The kernel lse_backward launches for back-to-back rows of N elements
    of eb bytes from a 16-byte aligned base into a dx of the same layout (the
    library's choice for that layout)."""
    epv = 16 // eb
    if N * eb % 16 == 0:  # every row on a 16-byte boundary
        return "lse_backward_small_kernel" if -(-N // epv) <= 8 else "lse_backward_kernel"
    if N >= epv and N * eb <= 16384:
        return "lse_backward_flat_kernel"
    if N // epv >= 4:
        return "lse_backward_kernel"  # head and tail peeled
    return "lse_backward_small_kernel" if N <= 4 else "lse_backward_kernel"  # element slots


def ncu_traffic(workload_key: str, plan: dict, op: str = "forward") -> float | None:
    """DRAM bytes per launch of the main kernel from the committed ncu record,
    or None when there is none for this workload, op and plan, or when the
    files that define the kernel changed since the capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)["entries"]
    except (OSError, KeyError, ValueError):
        return None
    for e in entries:
        if e.get("workload") != workload_key or e.get("op", "forward") != op:
            continue
        if e.get("path") != plan.get("path"):
            continue
        if any(k in plan and e.get(k) != plan[k] for k in ("grid", "threads")):
            continue
        try:
            if kernel_source_hash(e["sources"]) != e["source_hash"]:
                continue
        except (KeyError, OSError):
            continue
        return float(e["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self) -> dict:
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle, as it stands, on a bounded sample.
# ---------------------------------------------------------------------------
def time_oracle(x: np.ndarray, w: wl.Workload, budget_s: float, op: str = "forward") -> dict:
    import oracle

    rows = x.shape[0]
    if op == "logprob":
        t = np.random.default_rng(w.seed + 1).integers(0, w.N, rows)
        fn = lambda: oracle.token_logprob(x, t, w.dtype)  # noqa: E731
        bytes_per_row = w.N * w.elem_bytes + 12
    elif op == "backward":
        lse = oracle.lse(x, w.dtype)
        g = np.ones(rows)
        fn = lambda: oracle.backward(x, lse, g, w.dtype)  # noqa: E731
        bytes_per_row = 2 * w.N * w.elem_bytes + 8
    else:
        fn = lambda: oracle.lse(x, w.dtype)  # noqa: E731
        bytes_per_row = w.N * w.elem_bytes + 4
    oracle.lse(x[:1], w.dtype)  # load / build outside the timing
    rows_done, elapsed, reps = 0, 0.0, 0
    t0 = time.perf_counter()
    while True:
        fn()
        rows_done += rows
        reps += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= budget_s:
            break
    gbs = rows_done * bytes_per_row / elapsed / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "host": host_info(),
            "sample": f"{reps} pass(es) of the oracle's {OP_NAMES[op]} over {rows} rows x "
                      f"{w.N} {w.dtype} of the workload ({elapsed:.1f} s single-threaded)",
            "seconds": elapsed, "rows": rows_done}


def time_oracle_columns(x3: np.ndarray, cw, budget_s: float, op: str = "columns") -> dict:
    """The oracle's strided value (or its gradient) over the first slices of a
    column workload."""
    import oracle

    A = max(1, min(cw.A, int(budget_s / 4 / max(cw.R * cw.C * 8e-9, 1e-9))))
    sample = np.ascontiguousarray(x3[:A]).reshape(-1)
    args = (cw.dtype, A, cw.R, cw.C, cw.R * cw.C, cw.C)
    if op == "columns_backward":
        lse = oracle.lse_strided(sample, *args)
        g = np.ones((A, cw.C))
        fn = lambda: oracle.backward_strided(sample, *args, lse, g)  # noqa: E731
        bytes_per = A * (2 * cw.R * cw.C * cw.elem_bytes + cw.C * 8)
    else:
        fn = lambda: oracle.lse_strided(sample, *args)  # noqa: E731
        bytes_per = A * (cw.R * cw.C * cw.elem_bytes + cw.C * 4)
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= budget_s:
            break
    return {"value": reps * bytes_per / elapsed / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle", "host": host_info(),
            "sample": f"{reps} pass(es) of the oracle's {OP_NAMES[op]} over {A} of {cw.A} slices "
                      f"[{cw.R} x {cw.C}] ({elapsed:.1f} s single-threaded)",
            "seconds": elapsed}


def host_info() -> dict:
    """CPU model and logical core count of the machine the oracle runs on."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"cpu": model or platform.processor() or platform.machine(),
            "arch": platform.machine(), "nproc": os.cpu_count()}


def oracle_sample_rows(w: wl.Workload, target_s: float) -> int:
    """Rows of the workload that take roughly target_s of oracle time (~5 ns/elem)."""
    per_row = w.N * 5e-9
    return int(max(1, min(w.B, target_s / max(per_row, 1e-9))))


# ---------------------------------------------------------------------------
# The reference arm: the oracle as the comparison program.
# ---------------------------------------------------------------------------
REFERENCE_BUDGET_S = 60.0  # oracle seconds for a whole --impl reference run


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    # Each step is a bounded sample, sized so that the whole run (the steps
    # plus the warm-up steps, an eighth of a step each) takes about a minute
    # of oracle time whatever --steps is (at most 4 s per step).
    per_step_s = min(4.0, REFERENCE_BUDGET_S / (args.steps + args.warmup / 8))
    import oracle

    probe = wl.generate(args.workload, B=min(w.B, max(1, oracle_sample_rows(w, 0.05))))
    oracle.lse(probe[:1], w.dtype)
    t0 = time.perf_counter()
    oracle.lse(probe, w.dtype)
    per_row = max((time.perf_counter() - t0) / len(probe), 1e-9)  # this host's oracle speed
    rows = int(max(1, min(w.B, per_step_s / per_row)))
    x = wl.generate(args.workload, B=rows)
    for _ in range(args.warmup):
        oracle.lse(x[: max(1, rows // 8)], w.dtype)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.lse(x, w.dtype)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    bytes_per_step = rows * (w.N * w.elem_bytes + 4)
    gbs = bytes_per_step * len(times) / total / 1e9
    sample = (f"each step: {rows} of the workload's {w.B} rows ({w.N} {w.dtype} each), "
              f"fp64 oracle single-threaded")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": w.B, "N": w.N, "input_dtype": w.dtype,
                   "rows_per_step": rows, "recipe": w.recipe},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_info()},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# The native arm.
# ---------------------------------------------------------------------------
def to_torch(x: np.ndarray, dtype: str):
    import torch

    if dtype == "f32":
        return torch.from_numpy(x)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(x.view(np.int16)).view(tdt)


def run_native(args) -> None:
    import torch
    import torch.distributed as dist

    rank, world, local_rank = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from log_sum_exp_gb300 import build as lse_build
    lse_build.build()
    import log_sum_exp_gb300 as L

    if args.op in COLUMN_OPS:
        cw = wl.COLUMN_WORKLOADS[args.workload]
        x_host = wl.generate_columns(args.workload, seed=cw.seed + 7919 * rank)
        # Seen as B = A*C outputs of R-long strided reductions.
        w = wl.Workload(cw.key, cw.index, cw.A * cw.C, cw.R, cw.dtype, cw.recipe)
    else:
        cw = None
        w = wl.WORKLOADS[args.workload]
        x_host = wl.generate(args.workload, seed=rank_seed(w, rank))
    xt_host = to_torch(x_host, w.dtype)
    in_bytes = w.B * w.N * w.elem_bytes
    # Rotate over enough copies that consecutive steps never find their rows in L2.
    copies = max(1, -(-3 * L2_BYTES // max(in_bytes, 1)))
    copies = min(copies, 64)
    xs = [xt_host.to(dev) for _ in range(copies)]
    outs = [torch.empty(w.B, dtype=torch.float32, device=dev) for _ in range(copies)]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    dt = w.dtype
    ptrs = [(t.data_ptr(), o.data_ptr()) for t, o in zip(xs, outs)]
    op_name = args.op
    # A forced plan (--plan) is resolved by its first call and then reused.
    req = L._binding._as_plan(args.plan) if args.plan else None
    if op_name == "forward":
        if req is None:
            plan = L.lse_plan_query(xs[0])
        else:
            plan = L.lse_forward_plan_ptr(ptrs[0][0], dt, w.B, w.N, w.N, ptrs[0][1], sh,
                                          req).as_dict()
        bytes_per_step = in_bytes + w.write_bytes

        def step(i, evb=0, eve=0):
            xp, op = ptrs[i % copies]
            L.lse_forward_plan_ptr(xp, dt, w.B, w.N, w.N, op, sh, req, evb, eve)
    elif op_name == "forward16":
        plan = L.lse_forward16_ptr(ptrs[0][0], dt, w.B, w.N, w.N, ptrs[0][1], sh, req).as_dict()
        bytes_per_step = in_bytes + w.write_bytes

        def step(i, evb=0, eve=0):
            xp, op = ptrs[i % copies]
            L.lse_forward16_ptr(xp, dt, w.B, w.N, w.N, op, sh, req)
    elif op_name == "logprob":
        # Targets drawn once per copy; only the log-probabilities are written.
        rng = np.random.default_rng(w.seed + 1)
        tgts = [torch.from_numpy(rng.integers(0, w.N, w.B).astype(np.int64)).to(dev)
                for _ in range(copies)]
        plan = L.lse_token_logprob_ptr(ptrs[0][0], dt, w.B, w.N, w.N, tgts[0].data_ptr(),
                                       ptrs[0][1], 0, sh, req).as_dict()
        bytes_per_step = in_bytes + 8 * w.B + 4 * w.B

        def step(i, evb=0, eve=0):
            xp, op = ptrs[i % copies]
            L.lse_token_logprob_ptr(xp, dt, w.B, w.N, w.N, tgts[i % copies].data_ptr(), op, 0, sh,
                                    req)
    elif op_name == "columns":
        A, R, C = cw.A, cw.R, cw.C
        plan = L.lse_forward_strided_ptr(ptrs[0][0], dt, A, R, C, R * C, C, ptrs[0][1], sh,
                                         req).as_dict()
        bytes_per_step = in_bytes + w.write_bytes

        def step(i, evb=0, eve=0):
            xp, op = ptrs[i % copies]
            L.lse_forward_strided_ptr(xp, dt, A, R, C, R * C, C, op, sh, req)
    elif op_name == "columns_backward":
        A, R, C = cw.A, cw.R, cw.C
        for t, o in ptrs:  # the saved forward values, one set per copy
            L.lse_forward_strided_ptr(t, dt, A, R, C, R * C, C, o, sh)
        gs = [torch.ones(A * C, dtype=torch.float32, device=dev) for _ in range(copies)]
        dxs = [torch.empty_like(x) for x in xs]
        plan = {"path": "columns_backward", "launches": 1}
        bytes_per_step = 2 * in_bytes + 8 * A * C

        def step(i, evb=0, eve=0):
            c = i % copies
            L.lse_backward_strided_ptr(ptrs[c][0], dt, A, R, C, R * C, C, ptrs[c][1],
                                       gs[c].data_ptr(), dxs[c].data_ptr(), R * C, C, sh)
    else:  # backward
        lses = [L.lse_forward(x) for x in xs]
        gs = [torch.ones(w.B, dtype=torch.float32, device=dev) for _ in range(copies)]
        dxs = [torch.empty_like(x) for x in xs]
        plan = {"path": "backward", "launches": 1, "kernel": backward_kernel(w.N, 4 if dt == "f32" else 2)}
        bytes_per_step = 2 * in_bytes + 8 * w.B

        def step(i, evb=0, eve=0):
            c = i % copies
            L.lse_backward_ptr(ptrs[c][0], dt, w.B, w.N, w.N, lses[c].data_ptr(), gs[c].data_ptr(),
                               dxs[c].data_ptr(), w.N, sh)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    K = args.steps
    # Every EVENT_EVERY-th timed step brackets its main kernel with events (the
    # roofline's launch duration); the other steps run back to back untouched.
    # A one-kernel plan needs no per-step events: its launches are the whole
    # timed region.  Multi-kernel plans sample the main kernel's duration.
    sampled = list(range(0, K, EVENT_EVERY)) \
        if plan["launches"] > 1 and op_name == "forward" else []
    kb = {i: torch.cuda.Event(enable_timing=True) for i in sampled}
    ke = {i: torch.cuda.Event(enable_timing=True) for i in sampled}
    for e in list(kb.values()) + list(ke.values()):
        e.record(stream)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        time.sleep(0.25)  # a clock sample before the timed region
        start.record(stream)
        for i in range(K):
            if i in kb:
                step(i, kb[i].cuda_event, ke[i].cuda_event)
            else:
                step(i)
        end.record(stream)
        torch.cuda.synchronize(dev)
        time.sleep(0.25)
    barrier(dev)
    ms_total = start.elapsed_time(end)
    kernel_ms = [kb[i].elapsed_time(ke[i]) for i in sampled]
    ms_total = reduce_max(ms_total, dev)
    ms_per_step = ms_total / K
    value = world * bytes_per_step / (ms_per_step * 1e-3) / 1e9

    # Graph-replayed µs/call (launch overhead removed), same step.
    graph_us = None
    if args.graph and op_name == "forward":
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream(dev)
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            L.lse_forward_plan(xs[0], plan=args.plan, out=outs[0])
        stream.wait_stream(s2)
        reps = 100
        with torch.cuda.graph(g):
            for i in range(reps):
                L.lse_forward_plan(xs[i % copies], plan=args.plan, out=outs[i % copies])
        g.replay()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(10):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        graph_us = 1e3 * t0.elapsed_time(t1) / (10 * reps)

    # End to end through the host entry point: H2D of x, compute, D2H of out.
    e2e = None
    if op_name == "forward":
        e2e_steps = max(1, min(K, args.e2e_steps))
        x_pinned = xt_host.pin_memory()
        L.lse_forward_host(x_pinned)  # warm-up
        torch.cuda.synchronize(dev)
        barrier(dev)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            res = L.lse_forward_host(x_pinned)
        e2e_s = reduce_max(time.perf_counter() - t0, dev)
        assert res.shape == (w.B,)
        e2e = {"value": world * bytes_per_step * e2e_steps / e2e_s / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": w.write_bytes,
               "steps": e2e_steps,
               "call": "lse_forward_host on page-locked host x and out: the kernel "
                       "streams x over NVLink-C2C in place (zero copy), writes out in place"}

    if rank != 0:
        return
    peak, peak_src = measured_peaks()
    if kernel_ms:
        kmean_ms = sum(kernel_ms) / len(kernel_ms)
        kmed_ms = statistics.median(kernel_ms)
        timing = (f"CUDA events around the main kernel on every {EVENT_EVERY}th timed step "
                  f"({len(kernel_ms)} launches); includes the launch latency they bracket")
    else:
        kmean_ms = kmed_ms = ms_per_step
        timing = (f"one-kernel plan: CUDA events around the {K} back-to-back launches of the "
                  f"timed region, divided by {K}") if plan["launches"] == 1 else \
                 (f"{plan['launches']} kernels per step: CUDA events around the {K} steps of the "
                  f"timed region, divided by {K} (main kernel and merge together)")
    achieved = bytes_per_step / (kmean_ms * 1e-3) / 1e9
    main_kernel = {"subwarp": "lse_subwarp_kernel", "rowtile": "lse_rowtile_kernel",
                   "cta": "lse_segment_kernel",
                   "split": "lse_segment_kernel", "empty": "fill_neg_inf_kernel",
                   "backward": plan.get("kernel"), "columns_warp": "lse_cols_kernel",
                   "columns_cta": "lse_cols_kernel",
                   "columns_backward": "lse_backward_strided_kernel"}[plan["path"]]
    if plan["path"] == "rowtile" and plan.get("slots_per_lane") == 0:
        main_kernel = "lse_rowtile_any_kernel"  # rows of any width
    traffic = ncu_traffic(args.workload, plan, op_name)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": main_kernel,
                "peak_source": peak_src,
                "algorithmic_bytes_per_launch": bytes_per_step,
                "kernel_us_mean": 1e3 * kmean_ms,
                "kernel_us_median": 1e3 * kmed_ms,
                "kernel_timing": timing}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        if op_name in COLUMN_OPS:
            cpu = time_oracle_columns(x_host, cw, args.cpu_seconds, op_name)
        else:
            rows = oracle_sample_rows(w, args.cpu_seconds / 4)
            cpu = time_oracle(x_host[:rows], w, args.cpu_seconds, op_name)
    metric = METRIC if op_name == "forward" else f"{METRIC} [{OP_NAMES[op_name]}]"
    line = {
        "metric": metric, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 sums, bf16 exponentials" if op_name == "forward16" else "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "op": op_name, "B": w.B, "N": w.N,
                   **({"A": cw.A, "R": cw.R, "C": cw.C} if cw else {}),
                   "input_dtype": w.dtype, "row_stride": w.N, "recipe": w.recipe, "plan": plan,
                   "bytes_per_step": bytes_per_step,
                   "l2": f"inputs larger than L2: {copies} rotating copies of "
                         f"{in_bytes / 1e6:.1f} MB (L2 {L2_BYTES / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}, rows independent, no collective"},
        "us_per_call": 1e3 * ms_per_step,
        "pct_of_peak": 100.0 * value / peak,
        # x alone (the per-row outputs, targets or dx left out), and against
        # the public HBM3e figure rather than the measured copy peak.
        "read_gbs": world * in_bytes / (ms_per_step * 1e-3) / 1e9,
        "pct_of_spec_8tbs": 100.0 * value / SPEC_HBM_GBS,
        "us_per_call_graph": graph_us,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * plan["launches"],
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=list(wl.WORKLOADS) + list(wl.COLUMN_WORKLOADS),
                    default=None, help=f"default {DEFAULT_WORKLOAD} ({DEFAULT_COLUMNS} for "
                                       f"--op columns)")
    ap.add_argument("--op", choices=["forward", "forward16", "logprob", "backward", "columns",
                                     "columns_backward"],
                    default="forward",
                    help="row value (default), fused token log-probability, backward, or the "
                         "value over a non-last dimension (column workloads)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="skip the CUDA-graph replay timing (us_per_call_graph)")
    ap.add_argument("--plan", type=json.loads, default=None,
                    help='forced plan as JSON (fields of lse_plan, path by name), e.g. '
                         '{"path": "subwarp"} or, for --op columns, {"path": "columns_cta"}')
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print(f"bench.py: --warmup {args.warmup} raised to 3 (at least 3 warm-up steps)",
              file=sys.stderr)
        args.warmup = 3
    if args.workload is None:
        args.workload = DEFAULT_COLUMNS if args.op in COLUMN_OPS else DEFAULT_WORKLOAD
    if (args.op in COLUMN_OPS) != (args.workload in wl.COLUMN_WORKLOADS):
        ap.error("--op columns / columns_backward run the column workloads, the other ops "
                 "the row workloads")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
