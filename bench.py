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
    """nvidia-smi clocks and throttle reasons sampled every 100 ms, each sample
    with its timestamp so a summary can keep the samples of one window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

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

    @staticmethod
    def parse(line: str):
        """(unix time, sm MHz, max sm MHz, active throttle reasons) of one
        sample line, or None."""
        import datetime

        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            return None
        try:
            t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, smax = float(parts[2]), float(parts[3])
        except ValueError:
            return None
        reasons = [n for n, f in zip(ClockSampler.REASONS, parts[6:10])
                   if f.lower().startswith("active")]
        return t, sm, smax, reasons

    def summary(self, t_from: float | None = None, t_to: float | None = None) -> dict:
        """Median SM clock, max clock and throttle reasons over the samples
        taken in [t_from, t_to] (every sample when none falls in it)."""
        samples = [s for s in map(self.parse, self.lines) if s is not None]
        inside = [s for s in samples if (t_from is None or s[0] >= t_from) and
                  (t_to is None or s[0] <= t_to)]
        chosen = inside or samples
        if not chosen:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(s[1] for s in chosen),
                "sm_max_mhz": max(s[2] for s in chosen),
                "reasons": sorted({r for s in chosen for r in s[3]}), "samples": len(chosen),
                "samples_in_window": len(inside)}


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
# Host logic of the timing (also exercised by the CPU tests).
# ---------------------------------------------------------------------------
ROTATION_BYTES_MAX = 4 << 30  # device bytes the rotating input copies may take
CONFIG_STEPS_MIN = 200        # timed calls per config in per_config (>= 200 calls)
CONFIG_ORACLE_S = 2.0         # oracle seconds per config in per_config
CONFIG_BLOCKS = 4             # event blocks per config region (3 events inside 200+ calls)
REPEATS = 5                   # clean K-step regions repeated after the headline region
CLOCK_PROBE_S = 0.4           # the same step, untimed, after the region: clocks under load
SWEEP_BYTES = 512 << 20       # input bytes per step of the throughput-vs-N sweep
SWEEP_N = [16, 31, 32, 33, 64, 100, 128, 129, 256, 257, 300, 512, 520, 1000, 1024, 1025,
           2048, 4096, 4097, 8192, 16383, 16384, 32000, 32768, 50257, 65536, 128256, 262144,
           1048576, 4194304, 16777216]
COLS_SWEEP_BYTES = 256 << 20  # input bytes per call of the column sweep
COLS_SWEEP_R = [2, 8, 64, 512, 4096]
COLS_SWEEP_C = [64, 128, 192, 1000, 1024, 16384]


def rotation_copies(in_bytes: int, l2_bytes: int = L2_BYTES,
                    max_bytes: int = ROTATION_BYTES_MAX) -> int:
    """Input copies to rotate over so that each step reads rows that at least
    3x the L2 capacity of other copies' traffic has passed since (inputs
    larger than L2), within max_bytes of device memory."""
    if in_bytes <= 0:
        return 1
    want = -(-3 * l2_bytes // in_bytes)
    return int(max(1, min(want, max_bytes // in_bytes)))


def block_bounds(K: int, blocks: int) -> list[int]:
    """Step indices 0 = b_0 < b_1 < ... < b_n = K cutting K steps into
    min(blocks, K) nearly equal blocks."""
    n = max(1, min(blocks, K))
    return [round(i * K / n) for i in range(n + 1)]


def block_stats(bounds: list[int], block_ms: list[float]) -> dict:
    """µs per step of each block of back-to-back steps, their median, and the
    means over the first and the second half of the blocks (by steps)."""
    if not block_ms:
        return {}
    steps = [b - a for a, b in zip(bounds, bounds[1:])]
    per = [1e3 * t / n for t, n in zip(block_ms, steps)]
    h = len(per) // 2

    def mean(lo, hi):
        n = sum(steps[lo:hi])
        return 1e3 * sum(block_ms[lo:hi]) / n

    first, second = (mean(0, h), mean(h, len(per))) if h else (per[0], per[0])
    return {"us_per_step_blocks": per, "us_median": statistics.median(per),
            "us_mean": 1e3 * sum(block_ms) / sum(steps),
            "us_mean_first_half": first, "us_mean_second_half": second,
            "steps": sum(steps), "blocks": len(per)}


def main_kernel_name(plan: dict) -> str:
    """The kernel that moves the bytes in a plan (the roofline's kernel)."""
    path = plan["path"]
    if path == "rowtile" and plan.get("slots_per_lane") == 0:
        return "lse_rowtile_any_kernel"  # rows of any width
    return {"subwarp": "lse_subwarp_kernel", "rowtile": "lse_rowtile_kernel",
            "cta": "lse_segment_kernel", "split": "lse_segment_kernel",
            "empty": "fill_neg_inf_kernel", "backward": plan.get("kernel"),
            "columns_warp": "lse_cols_kernel", "columns_cta": "lse_cols_kernel",
            "columns_short": "lse_cols_short_kernel",
            "columns_backward": "lse_backward_strided_kernel"}[path]


def sweep_shape(N: int, eb: int, total: int = SWEEP_BYTES) -> tuple[int, int]:
    """(B, N) of one sweep point: rows of N elements filling ~total bytes."""
    return max(1, total // (N * eb)), N


def columns_sweep_shape(R: int, C: int, eb: int, total: int = COLS_SWEEP_BYTES) -> int:
    """A of one column-sweep point: [A, R, C] filling ~total bytes (0: does not fit once)."""
    return total // (R * C * eb)


def columns_sweep_table(points: list[dict]) -> str:
    """Markdown table of column-sweep points (forward and backward)."""
    lines = ["| dtype | R | C | A | forward plan | forward µs | forward GB/s | frac | "
             "backward µs | backward GB/s | frac |",
             "|---|---|---|---|---|---|---|---|---|---|---|"]
    for q in points:
        p = q["plan"]
        desc = {"columns_warp": "warp", "columns_short": "short"}.get(p["path"], f"cta WT={p['lanes_per_row']}") + \
               (" elem" if p["vector_bytes"] == 1 else "") + (f" P={p['splits']}" if p["splits"] > 1 else "")
        lines.append(f"| {q['dtype']} | {q['R']} | {q['C']} | {q['A']} | {desc} | {q['fwd_us']:.2f} | "
                     f"{q['fwd_gbs']:.0f} | {q['fwd_frac']:.3f} | {q['bwd_us']:.2f} | "
                     f"{q['bwd_gbs']:.0f} | {q['bwd_frac']:.3f} |")
    return "\n".join(lines)


def sweep_table(points: list[dict]) -> str:
    """Markdown table of sweep points."""
    lines = ["| dtype | N | B | plan | µs / call (median) | GB/s | frac of measured |",
             "|---|---|---|---|---|---|---|"]
    for q in points:
        p = q["plan"]
        desc = p["path"]
        if p["path"] in ("cta", "split"):
            desc += f" T={p['threads']}" + (f" P={p['splits']}" if p["splits"] > 1 else "")
        elif p["path"] == "subwarp":
            desc += f" G={p['lanes_per_row']} V={p['slots_per_lane']}"
        elif p["path"] == "rowtile":
            desc += f" {'any-width' if p['slots_per_lane'] == 0 else str(p['slots_per_lane']) + ' vec'}" \
                    + (f" G={p['lanes_per_row']}" if p["slots_per_lane"] == 0 else "")
        lines.append(f"| {q['dtype']} | {q['N']} | {q['B']} | {desc} | {q['us_median']:.2f} | "
                     f"{q['gbs']:.0f} | {q['frac']:.3f} |")
    return "\n".join(lines)


# ---------------------------------------------------------------------------
# The native arm.
# ---------------------------------------------------------------------------
def to_torch(x: np.ndarray, dtype: str):
    import torch

    if dtype == "f32":
        return torch.from_numpy(x)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(x.view(np.int16)).view(tdt)


def timed_steps(step, K: int, stream, blocks: int = 1, event_every: dict | None = None,
                first: int = 0):
    """Run step(first .. first+K-1) back to back, with CUDA events only at the
    block bounds (block_bounds(K, blocks)): an event between two launches
    removes their programmatic overlap (measured: +4.5 µs on a 40 µs step), so
    a one-block region has none inside it.  Returns (bounds, total ms, ms per
    block).  event_every maps a step index to (begin, end) events handed to
    the step (its main kernel)."""
    import torch

    bounds = block_bounds(K, blocks)
    evs = [torch.cuda.Event(enable_timing=True) for _ in bounds]
    evs[0].record(stream)
    b = 1
    for i in range(K):
        if event_every and i in event_every:
            step(first + i, event_every[i][0].cuda_event, event_every[i][1].cuda_event)
        else:
            step(first + i)
        if i + 1 == bounds[b]:
            evs[b].record(stream)
            b += 1
    torch.cuda.synchronize()
    per = [evs[j].elapsed_time(evs[j + 1]) for j in range(len(bounds) - 1)]
    return bounds, evs[0].elapsed_time(evs[-1]), per


def graph_us_per_call(L, xs, outs, plan_req, stream, dev, reps: int = 100) -> float:
    """lse_forward replayed from a CUDA graph of `reps` calls over the rotating
    copies: µs per call with the launch overhead removed."""
    import torch

    g = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream(dev)
    s2.wait_stream(stream)
    with torch.cuda.stream(s2):
        L.lse_forward_plan(xs[0], plan=plan_req, out=outs[0])
    stream.wait_stream(s2)
    with torch.cuda.graph(g):
        for i in range(reps):
            L.lse_forward_plan(xs[i % len(xs)], plan=plan_req, out=outs[i % len(xs)])
    g.replay()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(10):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    return 1e3 * t0.elapsed_time(t1) / (10 * reps)


def measure_config(L, key: str, rank: int, dev, stream, steps: int, peak: float,
                   graph: bool = True) -> tuple[dict, np.ndarray]:
    """One row workload through lse_forward: µs per call (per-step CUDA events,
    inputs rotated past L2), GB/s and fraction of the measured peak, and the
    CUDA-graph µs per call.  Returns (entry, a host sample for the oracle)."""
    import torch

    w = wl.WORKLOADS[key]
    x_host = wl.generate(key, seed=rank_seed(w, rank))
    in_bytes = w.B * w.N * w.elem_bytes
    copies = rotation_copies(in_bytes)
    xt = to_torch(x_host, w.dtype)
    xs = [xt.to(dev) for _ in range(copies)]
    outs = [torch.empty(w.B, dtype=torch.float32, device=dev) for _ in range(copies)]
    ptrs = [(t.data_ptr(), o.data_ptr()) for t, o in zip(xs, outs)]
    sh = stream.cuda_stream
    plan = L.lse_plan_query(xs[0])

    def step(i, evb=0, eve=0):
        xp, op = ptrs[i % copies]
        L.lse_forward_plan_ptr(xp, w.dtype, w.B, w.N, w.N, op, sh, None, evb, eve)

    for i in range(10):
        step(i)
    torch.cuda.synchronize(dev)
    K = max(steps, CONFIG_STEPS_MIN)
    bounds, total_ms, per = timed_steps(step, K, stream, blocks=CONFIG_BLOCKS)
    stats = block_stats(bounds, per)
    bytes_per_call = in_bytes + w.write_bytes
    us_mean = 1e3 * total_ms / K
    entry = {"workload": key, "B": w.B, "N": w.N, "input_dtype": w.dtype,
             "plan": {k: plan[k] for k in ("path", "threads", "splits", "grid", "lanes_per_row",
                                           "slots_per_lane", "launches")},
             "kernel": main_kernel_name(plan), "bytes_per_call": bytes_per_call,
             "us_per_call": us_mean, "us_median_of_blocks": stats["us_median"],
             "us_mean_first_half": stats["us_mean_first_half"],
             "us_mean_second_half": stats["us_mean_second_half"], "calls": K,
             "timing": f"CUDA events at {CONFIG_BLOCKS + 1} points of {K} back-to-back calls "
                       f"(inputs in HBM); us_per_call = total / {K}",
             "gbs": bytes_per_call / (us_mean * 1e-6) / 1e9,
             "frac": bytes_per_call / (us_mean * 1e-6) / 1e9 / peak,
             "traffic": ncu_traffic(key, plan, "forward"),
             "l2": f"{copies} rotating copies of {in_bytes / 1e6:.1f} MB (L2 {L2_BYTES / 1e6:.0f} MB)"}
    entry["us_per_call_graph"] = graph_us_per_call(L, xs, outs, None, stream, dev) if graph else None
    del xs, outs
    torch.cuda.empty_cache()
    rows = max(1, min(w.B, oracle_sample_rows(w, CONFIG_ORACLE_S / 4)))
    return entry, x_host[:rows].copy()


def run_sweep(args) -> None:
    """Throughput of lse_forward against the row length N at ~512 MB of input
    per call, f32 and bf16, automatic plan: one JSON line per point, then a
    markdown table."""
    import torch

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from log_sum_exp_gb300 import build as lse_build
    lse_build.build()
    import log_sum_exp_gb300 as L

    peak, _ = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    gen = torch.Generator(device=dev)
    points = []
    for dtype in ("f32", "bf16"):
        eb = 4 if dtype == "f32" else 2
        tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        for N in SWEEP_N:
            B, N = sweep_shape(N, eb)
            gen.manual_seed(wl.SEED_BASE + 100 + N)
            # Two copies of ~512 MB each: every call reads rows absent from L2.
            xs = [(3.0 * torch.randn(B, N, device=dev, generator=gen)).to(tdt) for _ in range(2)]
            outs = [torch.empty(B, dtype=torch.float32, device=dev) for _ in range(2)]
            plan = L.lse_plan_query(xs[0])

            def step(i, evb=0, eve=0):
                L.lse_forward_plan_ptr(xs[i % 2].data_ptr(), dtype, B, N, N, outs[i % 2].data_ptr(),
                                       sh, None)

            for i in range(5):
                step(i)
            torch.cuda.synchronize(dev)
            bounds, _, per = timed_steps(step, args.sweep_steps, stream, blocks=3)
            st = block_stats(bounds, per)
            nbytes = B * N * eb + 4 * B
            q = {"dtype": dtype, "N": N, "B": B, "plan": plan, "us_median": st["us_median"],
                 "gbs": nbytes / (st["us_median"] * 1e-6) / 1e9}
            q["frac"] = q["gbs"] / peak
            points.append(q)
            print(json.dumps(q), flush=True)
            del xs, outs
            torch.cuda.empty_cache()
    print(sweep_table(points), flush=True)


def run_sweep_columns(args) -> None:
    """Throughput of lse_forward_strided and lse_backward_strided over R (the
    reduced dimension) and C at ~256 MB of input per call, f32 and bf16,
    automatic plan: one JSON line per point, then a markdown table."""
    import torch

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from log_sum_exp_gb300 import build as lse_build
    lse_build.build()
    import log_sum_exp_gb300 as L

    peak, _ = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    gen = torch.Generator(device=dev)
    points = []
    for dtype in ("f32", "bf16"):
        eb = 4 if dtype == "f32" else 2
        tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        for R in COLS_SWEEP_R:
            for C in COLS_SWEEP_C:
                A = columns_sweep_shape(R, C, eb)
                if A < 1:
                    continue
                gen.manual_seed(wl.SEED_BASE + 200 + R + C)
                # Two copies: every call reads rows absent from L2.
                xs = [(3.0 * torch.randn(A, R, C, device=dev, generator=gen)).to(tdt) for _ in range(2)]
                outs = [torch.empty(A, C, dtype=torch.float32, device=dev) for _ in range(2)]
                grad = torch.ones(A, C, dtype=torch.float32, device=dev)
                dx = torch.empty_like(xs[0])
                plan = L.lse_forward_strided_ptr(xs[0].data_ptr(), dtype, A, R, C, R * C, C,
                                                 outs[0].data_ptr(), sh).as_dict()

                def fwd(i, evb=0, eve=0):
                    L.lse_forward_strided_ptr(xs[i % 2].data_ptr(), dtype, A, R, C, R * C, C,
                                              outs[i % 2].data_ptr(), sh)

                def bwd(i, evb=0, eve=0):
                    L.lse_backward_strided_ptr(xs[i % 2].data_ptr(), dtype, A, R, C, R * C, C,
                                               outs[i % 2].data_ptr(), grad.data_ptr(),
                                               dx.data_ptr(), R * C, C, sh)

                q = {"dtype": dtype, "R": R, "C": C, "A": A, "plan": plan}
                for name, step, nbytes in (("fwd", fwd, A * R * C * eb + 4 * A * C),
                                           ("bwd", bwd, 2 * A * R * C * eb + 8 * A * C)):
                    for i in range(5):
                        step(i)
                    torch.cuda.synchronize(dev)
                    bounds, _, per = timed_steps(step, args.sweep_steps, stream, blocks=3)
                    us = block_stats(bounds, per)["us_median"]
                    q[name + "_us"] = us
                    q[name + "_gbs"] = nbytes / (us * 1e-6) / 1e9
                    q[name + "_frac"] = q[name + "_gbs"] / peak
                points.append(q)
                print(json.dumps(q), flush=True)
                del xs, outs, grad, dx
                torch.cuda.empty_cache()
    print(columns_sweep_table(points), flush=True)


def run_native(args) -> None:
    import torch
    import torch.distributed as dist

    rank, world, local_rank = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    clocks = ClockSampler(local_rank)
    clocks.__enter__()

    from log_sum_exp_gb300 import build as lse_build
    lse_build.build()
    import log_sum_exp_gb300 as L

    peak, peak_src = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # The five row workloads, each through lse_forward (one GPU, rank 0).
    per_config, config_samples = None, {}
    if args.op == "forward" and args.per_config and world == 1:
        per_config = {}
        for key in wl.ORDER:
            entry, sample = measure_config(L, key, rank, dev, stream, args.steps, peak, args.graph)
            per_config[key] = entry
            config_samples[key] = sample

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
    copies = rotation_copies(in_bytes)
    xs = [xt_host.to(dev) for _ in range(copies)]
    outs = [torch.empty(w.B, dtype=torch.float32, device=dev) for _ in range(copies)]
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

    # W untimed warm-up steps right before the timed region (no idle gap).
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    K = args.steps
    # One clean region: events only before the first step and after the last
    # (an event between two launches would cost them their programmatic
    # overlap).  For a two-kernel row-value plan, every EVENT_EVERY-th step
    # also brackets its main kernel (the roofline's launch duration).
    sampled = list(range(0, K, EVENT_EVERY)) \
        if plan["launches"] > 1 and op_name == "forward" else []
    kev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for i in sampled}
    for pair in kev.values():  # create the events (torch does so lazily, on a first record)
        for e in pair:
            e.record(stream)
    barrier(dev)
    torch.cuda.synchronize(dev)
    t_region = time.time()
    _, ms_total, _ = timed_steps(step, K, stream, 1, kev)
    t_region_end = time.time()
    barrier(dev)
    # The same K-step region repeated (clean): start-up against steady state.
    repeats = [timed_steps(step, K, stream, 1, None, (r + 1) * K)[1] for r in range(REPEATS)]
    # Clocks under the same load: the same step, untimed, for CLOCK_PROBE_S after the region.
    t0 = time.perf_counter()
    i = (REPEATS + 1) * K
    while time.perf_counter() - t0 < CLOCK_PROBE_S:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    t_probe_end = time.time()
    kernel_ms = [kev[i][0].elapsed_time(kev[i][1]) for i in sampled]
    ms_total = reduce_max(ms_total, dev)
    ms_per_step = ms_total / K
    value = world * bytes_per_step / (ms_per_step * 1e-3) / 1e9
    region_us = [1e3 * ms_per_step] + [1e3 * t / K for t in repeats]
    steps_summary = {"region_means_us": region_us, "median_of_regions_us": statistics.median(region_us),
                     "about": f"the timed region, then the same {K} steps {REPEATS} more times, "
                              f"each region clean (events at its ends only)"}

    # Graph-replayed µs/call (launch overhead removed), same step.
    graph_us = None
    if args.graph and op_name == "forward":
        graph_us = graph_us_per_call(L, xs, outs, args.plan, stream, dev)

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
    clocks.__exit__(None, None, None)

    if rank != 0:
        return
    if kernel_ms:
        kmean_ms = sum(kernel_ms) / len(kernel_ms)
        kmed_ms = statistics.median(kernel_ms)
        timing = (f"CUDA events around the main kernel on every {EVENT_EVERY}th timed step "
                  f"({len(kernel_ms)} launches); includes the launch latency they bracket")
    else:
        kmean_ms = ms_per_step
        kmed_ms = steps_summary["median_of_regions_us"] * 1e-3
        timing = (f"one-kernel plan: CUDA events around the {K} back-to-back launches of the "
                  f"timed region, divided by {K}; median over that region and {REPEATS} "
                  f"repeats of it") if plan["launches"] == 1 else \
                 (f"{plan['launches']} kernels per step: CUDA events around the {K} steps of the "
                  f"timed region, divided by {K} (main kernel and merge together); median over "
                  f"that region and {REPEATS} repeats of it")
    achieved = bytes_per_step / (kmean_ms * 1e-3) / 1e9
    main_kernel = main_kernel_name(plan)
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
        if per_config is not None:
            for key, entry in per_config.items():
                entry["cpu_baseline"] = time_oracle(config_samples[key], wl.WORKLOADS[key],
                                                    CONFIG_ORACLE_S)
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
        "step_times": steps_summary,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * plan["launches"],
        "clocks": {**clocks.summary(t_region - 0.05, t_probe_end + 0.05),
                   "window": f"the {1e3 * (t_region_end - t_region):.1f} ms timed region and "
                             f"{CLOCK_PROBE_S} s of the same step right after it"},
    }
    if per_config is not None:
        line["per_config"] = per_config
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
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the per_config block (every row workload timed through "
                         "lse_forward before the headline step)")
    ap.add_argument("--sweep", action="store_true",
                    help="throughput against N at ~512 MB per call (f32, bf16): JSON lines "
                         "and a markdown table instead of the bench line")
    ap.add_argument("--sweep-columns", action="store_true",
                    help="throughput of the value over a non-last dimension and its backward "
                         "against R and C at ~256 MB per call (f32, bf16): JSON lines and a "
                         "markdown table instead of the bench line")
    ap.add_argument("--sweep-steps", type=int, default=30)
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
    elif args.sweep:
        run_sweep(args)
    elif args.sweep_columns:
        run_sweep_columns(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
