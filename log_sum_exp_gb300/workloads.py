"""Seeded synthetic inputs for the row-wise log-sum-exp.

This module only draws numbers: it holds none of the log-sum-exp arithmetic,
and both the CUDA path's tests/benchmark and the fp64 oracle read the arrays
it returns.  Every array comes from numpy's Philox counter-based generator
(Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11) keyed by
a fixed seed, filled in fixed slabs so the bits do not depend on memory size.

The five workloads stand in for the paper's GPU settings ("Speeding up
Log-Sum-Exp ...", Sec. 2.1/Fig. 1 for the (512, 128256) profile, Sec. 5.1 for
32K-256K vocabularies, Sec. 5.2 for probabilistic-circuit sum layers and
Sec. 5.3 for particle log-weights); the pages' own datasets and trained
weights are not used.
"""
from __future__ import annotations

import dataclasses

import numpy as np

SEED_BASE = 20261202
_SLAB_ELEMS = 1 << 22  # elements drawn per generator call


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    index: int
    B: int
    N: int
    dtype: str  # "f32" | "bf16" | "f16"
    recipe: str

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def read_bytes(self) -> int:
        return self.B * self.N * self.elem_bytes

    @property
    def write_bytes(self) -> int:
        return self.B * 4

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


WORKLOADS = {
    w.key: w for w in [
        Workload("small_64x4096_f32", 1, 64, 4096, "f32",
                 "x ~ N(0,1) i.i.d."),
        Workload("vocab_512x128256_f32", 2, 512, 128256, "f32",
                 "x = o_b + 3 z, z ~ N(0,1), o_b ~ U(-20,20) per row; one entry per row "
                 "(seeded column) set to o_b + 15"),
        Workload("vocab_8192x32000_bf16", 3, 8192, 32000, "bf16",
                 "x = 2 z, z ~ N(0,1) in f32; rows [0,B/4) shifted +1000, rows [B/4,B/2) "
                 "shifted -1000; rounded to bf16 (nearest-even)"),
        Workload("short_1048576x32_f32", 4, 1048576, 32, "f32",
                 "x ~ U(-30,0); each entry -inf with p=0.1; floor(B/1000) rows all -inf; "
                 "floor(B/1e5) other rows hold one NaN at a seeded column"),
        Workload("particles_16x16777216_f32", 5, 16, 16777216, "f32",
                 "x ~ U(-50,0]; one entry per row (seeded column) set to 0"),
    ]
}
ORDER = [k for k, _ in sorted(WORKLOADS.items(), key=lambda kv: kv[1].index)]


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def _fill_normal(rng: np.random.Generator, out: np.ndarray) -> None:
    flat = out.reshape(-1)
    for lo in range(0, flat.size, _SLAB_ELEMS):
        hi = min(flat.size, lo + _SLAB_ELEMS)
        rng.standard_normal(hi - lo, dtype=np.float32, out=flat[lo:hi])


def _fill_uniform01(rng: np.random.Generator, out: np.ndarray) -> None:
    flat = out.reshape(-1)
    for lo in range(0, flat.size, _SLAB_ELEMS):
        hi = min(flat.size, lo + _SLAB_ELEMS)
        rng.random(hi - lo, dtype=np.float32, out=flat[lo:hi])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest, ties to even); raw uint16 bits."""
    flat = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(flat.size, dtype=np.uint16)
    for lo in range(0, flat.size, _SLAB_ELEMS):
        hi = min(flat.size, lo + _SLAB_ELEMS)
        bits = flat[lo:hi].view(np.uint32)
        bias = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
        out[lo:hi] = ((bits + bias) >> np.uint32(16)).astype(np.uint16)
    return out.reshape(x.shape)


def generate(key: str, B: int | None = None, N: int | None = None,
             seed: int | None = None) -> np.ndarray:
    """The workload's input as a contiguous [B, N] array.

    f32 workloads return float32; bf16 workloads return the raw uint16 bits.
    ``B``/``N`` override the shape (same recipe, smaller or ragged sizes);
    ``seed`` overrides the workload's seed.
    """
    w = WORKLOADS[key]
    B = w.B if B is None else B
    N = w.N if N is None else N
    rng = _rng(w.seed if seed is None else seed)
    gen = _GENERATORS[w.index]
    return gen(rng, B, N)


def _gen_small(rng, B, N):
    x = np.empty((B, N), dtype=np.float32)
    _fill_normal(rng, x)
    return x


def _gen_vocab128k(rng, B, N):
    x = np.empty((B, N), dtype=np.float32)
    _fill_normal(rng, x)
    offset = rng.uniform(-20.0, 20.0, size=B).astype(np.float32)
    x *= np.float32(3.0)
    x += offset[:, None]
    if N > 0:
        cols = rng.integers(0, N, size=B)
        x[np.arange(B), cols] = offset + np.float32(15.0)
    return x


def _gen_vocab32k_bf16(rng, B, N):
    x = np.empty((B, N), dtype=np.float32)
    _fill_normal(rng, x)
    x *= np.float32(2.0)
    q = B // 4
    x[:q] += np.float32(1000.0)
    x[q:2 * q] -= np.float32(1000.0)
    return f32_to_bf16_bits(x)


def _gen_short(rng, B, N):
    x = np.empty((B, N), dtype=np.float32)
    _fill_uniform01(rng, x)
    x *= np.float32(-30.0)
    mask = np.empty((B, N), dtype=np.float32)
    _fill_uniform01(rng, mask)
    x[mask < np.float32(0.1)] = -np.inf
    del mask
    perm = rng.permutation(B)
    n_all_neg_inf = B // 1000
    n_nan = B // 100000
    x[perm[:n_all_neg_inf]] = -np.inf
    nan_rows = perm[n_all_neg_inf:n_all_neg_inf + n_nan]
    if N > 0 and nan_rows.size:
        x[nan_rows, rng.integers(0, N, size=nan_rows.size)] = np.nan
    return x


def _gen_particles(rng, B, N):
    x = np.empty((B, N), dtype=np.float32)
    _fill_uniform01(rng, x)
    x *= np.float32(-50.0)
    if N > 0:
        x[np.arange(B), rng.integers(0, N, size=B)] = np.float32(0.0)
    return x


_GENERATORS = {1: _gen_small, 2: _gen_vocab128k, 3: _gen_vocab32k_bf16, 4: _gen_short,
               5: _gen_particles}


@dataclasses.dataclass(frozen=True)
class ColumnWorkload:
    """x: [A, R, C]; the value is taken over R (a non-last dimension)."""
    key: str
    index: int
    A: int
    R: int
    C: int
    dtype: str
    recipe: str

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def read_bytes(self) -> int:
        return self.A * self.R * self.C * self.elem_bytes

    @property
    def write_bytes(self) -> int:
        return self.A * self.C * 4

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


COLUMN_WORKLOADS = {
    w.key: w for w in [
        ColumnWorkload("pcsum_512x64x1024_f32", 11, 512, 64, 1024, "f32",
                       "sum-layer log-weights: x[batch a, child r, node c] ~ U(-30,0), each entry "
                       "-inf with p=0.1; the value is over the 64 children of each node"),
        ColumnWorkload("columns_1x8192x16384_f32", 12, 1, 8192, 16384, "f32",
                       "column LSE of a tall matrix: x ~ N(0, 3^2) + per-column offset U(-20,20)"),
    ]
}


def generate_columns(key: str, A: int | None = None, R: int | None = None,
                     C: int | None = None, seed: int | None = None) -> np.ndarray:
    """A column workload's input as a contiguous [A, R, C] float32 array."""
    w = COLUMN_WORKLOADS[key]
    A = w.A if A is None else A
    R = w.R if R is None else R
    C = w.C if C is None else C
    rng = _rng(w.seed if seed is None else seed)
    x = np.empty((A, R, C), dtype=np.float32)
    if w.index == 11:
        _fill_uniform01(rng, x)
        x *= np.float32(-30.0)
        mask = np.empty_like(x)
        _fill_uniform01(rng, mask)
        x[mask < np.float32(0.1)] = -np.inf
    else:
        _fill_normal(rng, x)
        x *= np.float32(3.0)
        x += rng.uniform(-20.0, 20.0, size=(1, 1, C)).astype(np.float32)
    return x


def random_rows(B: int, N: int, dtype: str = "f32", seed: int = 0, scale: float = 4.0,
                shift: float = 0.0) -> np.ndarray:
    """Generic seeded rows ``shift + scale * z`` for edge-shape tests.

    f32 -> float32; bf16 -> raw uint16 bits (nearest-even); f16 -> float16.
    """
    rng = _rng(SEED_BASE + 1000 + seed)
    x = np.empty((B, N), dtype=np.float32)
    _fill_normal(rng, x)
    x *= np.float32(scale)
    x += np.float32(shift)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":
        return x.astype(np.float16)
    raise ValueError(dtype)
