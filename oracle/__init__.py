"""fp64 CPU oracle for the row-wise log-sum-exp.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA path never
calls it, and the two share no code: the oracle is the plain definition
``out[b] = log sum_n exp(x[b, n])`` written out in C (``lse_oracle.c``), single
threaded, in double precision.

Source: "Speeding up Log-Sum-Exp: Kernel Fusion at the Memory Wall, Integer
Arithmetic at the Compute Wall" -- Sec. 2.1 (the max-subtract recipe that
torch.logsumexp expands into its sub-kernels, Fig. 1) and Sec. 4 (accuracy is
measured against an FP64 baseline).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lse_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblse_oracle.so")

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """ctypes view of one compiled oracle library (the real one, or a test's mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_lse.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        lib.oracle_lse.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_void_p]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_token_logprob.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_token_logprob.restype = ctypes.c_int
        lib.oracle_lse_backward.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_lse_backward.restype = ctypes.c_int
        lib.oracle_lse_strided.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_void_p]
        lib.oracle_lse_strided.restype = ctypes.c_int
        lib.oracle_lse_backward_strided.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_lse_backward_strided.restype = ctypes.c_int
        self._lib = lib
        self.path = path

    def lse(self, x: np.ndarray, dtype: str = "f32", B: int | None = None,
            N: int | None = None, row_stride: int | None = None) -> np.ndarray:
        return _lse(self._lib, x, dtype, B, N, row_stride)

    def decode(self, x: np.ndarray, dtype: str) -> np.ndarray:
        return _decode(self._lib, x, dtype)

    def token_logprob(self, x: np.ndarray, target: np.ndarray, dtype: str = "f32",
                      row_stride: int | None = None, N: int | None = None):
        return _token_logprob(self._lib, x, target, dtype, row_stride, N)

    def backward(self, x: np.ndarray, lse: np.ndarray, grad: np.ndarray, dtype: str = "f32",
                 row_stride: int | None = None, N: int | None = None) -> np.ndarray:
        return _backward(self._lib, x, lse, grad, dtype, row_stride, N)

    def lse_strided(self, x: np.ndarray, dtype: str, A: int, R: int, C: int, stride_a: int,
                    stride_r: int) -> np.ndarray:
        return _lse_strided(self._lib, x, dtype, A, R, C, stride_a, stride_r)

    def backward_strided(self, x: np.ndarray, dtype: str, A: int, R: int, C: int,
                         stride_a: int, stride_r: int, lse: np.ndarray,
                         grad: np.ndarray) -> np.ndarray:
        return _backward_strided(self._lib, x, dtype, A, R, C, stride_a, stride_r, lse, grad)


def _load() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def lse(x: np.ndarray, dtype: str = "f32", B: int | None = None, N: int | None = None,
        row_stride: int | None = None) -> np.ndarray:
    """out[b] = log sum_n exp(x[b, n]) in float64 (see ``_lse``)."""
    return _load().lse(x, dtype, B, N, row_stride)


def decode(x: np.ndarray, dtype: str) -> np.ndarray:
    """The oracle's exact element decode (raw elements -> float64)."""
    return _load().decode(x, dtype)


def token_logprob(x: np.ndarray, target: np.ndarray, dtype: str = "f32",
                  row_stride: int | None = None, N: int | None = None):
    """(logprob, lse): logprob[b] = x[b, target[b]] - lse[b] in float64 (NaN for a
    target outside [0, N)).  ``x`` is 2-D [B, row_stride]; the first N columns
    are the row."""
    return _load().token_logprob(x, target, dtype, row_stride, N)


def backward(x: np.ndarray, lse: np.ndarray, grad: np.ndarray, dtype: str = "f32",
             row_stride: int | None = None, N: int | None = None) -> np.ndarray:
    """dx[b, n] = grad[b] * exp(x[b, n] - lse[b]) in float64, dense [B, N]."""
    return _load().backward(x, lse, grad, dtype, row_stride, N)


def lse_strided(x: np.ndarray, dtype: str, A: int, R: int, C: int, stride_a: int,
                stride_r: int) -> np.ndarray:
    """out[a, c] = log sum_r exp(x[a*stride_a + r*stride_r + c]) in float64, [A, C].

    ``x`` is a flat buffer of raw elements (float32, or 16-bit patterns)."""
    return _load().lse_strided(x, dtype, A, R, C, stride_a, stride_r)


def backward_strided(x: np.ndarray, dtype: str, A: int, R: int, C: int, stride_a: int,
                     stride_r: int, lse: np.ndarray, grad: np.ndarray) -> np.ndarray:
    """dx[a, r, c] = grad[a, c] * exp(x[a*stride_a + r*stride_r + c] - lse[a, c]) in
    float64, [A, R, C]: the gradient of lse_strided's value.  ``lse`` and ``grad``
    are [A, C]."""
    return _load().backward_strided(x, dtype, A, R, C, stride_a, stride_r, lse, grad)


def _backward_strided(lib, x, dtype, A, R, C, stride_a, stride_r, lse, grad):
    arr = _raw(x, dtype).reshape(-1)
    if A > 0 and R > 0 and C > 0:
        need = (A - 1) * stride_a + (R - 1) * stride_r + C
        if arr.size < need:
            raise ValueError(f"buffer of {arr.size} elements, need {need}")
    lse = np.ascontiguousarray(lse, dtype=np.float64).reshape(-1)
    grad = np.ascontiguousarray(grad, dtype=np.float64).reshape(-1)
    if lse.size != A * C or grad.size != A * C:
        raise ValueError("lse and grad hold one value per (a, c)")
    dx = np.empty((A, R, C), np.float64)
    if dx.size:
        rc = lib.oracle_lse_backward_strided(arr.ctypes.data, DTYPE_CODES[dtype], A, R, C,
                                             stride_a, stride_r, lse.ctypes.data,
                                             grad.ctypes.data, dx.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_lse_backward_strided rejected its arguments")
    return dx


def _lse_strided(lib, x, dtype, A, R, C, stride_a, stride_r):
    arr = _raw(x, dtype).reshape(-1)
    if A > 0 and R > 0 and C > 0:
        need = (A - 1) * stride_a + (R - 1) * stride_r + C
        if arr.size < need:
            raise ValueError(f"buffer of {arr.size} elements, need {need}")
    out = np.empty((A, C), np.float64)
    rc = lib.oracle_lse_strided(arr.ctypes.data if arr.size else None, DTYPE_CODES[dtype], A, R,
                                C, stride_a, stride_r, out.ctypes.data if out.size else None)
    if rc != 0:
        raise ValueError("oracle_lse_strided rejected its arguments")
    return out


def _shape2d(arr: np.ndarray, row_stride, N):
    if arr.ndim != 2:
        raise ValueError("expected a 2-D [B, row_stride] array")
    B = arr.shape[0]
    row_stride = arr.shape[1] if row_stride is None else row_stride
    N = row_stride if N is None else N
    if row_stride != arr.shape[1] or N > row_stride:
        raise ValueError("row_stride must equal the array's second dimension and N <= it")
    return B, N, row_stride


def _token_logprob(lib, x, target, dtype, row_stride, N):
    arr = _raw(x, dtype)
    B, N, row_stride = _shape2d(arr, row_stride, N)
    t = np.ascontiguousarray(target, dtype=np.int64).reshape(-1)
    if t.size != B:
        raise ValueError("one target per row")
    logprob = np.empty(B, np.float64)
    lse_out = np.empty(B, np.float64)
    rc = lib.oracle_token_logprob(arr.ctypes.data if arr.size else None, DTYPE_CODES[dtype], B, N,
                                  row_stride, t.ctypes.data if B else None,
                                  logprob.ctypes.data if B else None,
                                  lse_out.ctypes.data if B else None)
    if rc != 0:
        raise ValueError("oracle_token_logprob rejected its arguments")
    return logprob, lse_out


def _backward(lib, x, lse, grad, dtype, row_stride, N):
    arr = _raw(x, dtype)
    B, N, row_stride = _shape2d(arr, row_stride, N)
    lse = np.ascontiguousarray(lse, dtype=np.float64).reshape(-1)
    grad = np.ascontiguousarray(grad, dtype=np.float64).reshape(-1)
    if lse.size != B or grad.size != B:
        raise ValueError("one lse and one grad per row")
    dx = np.empty((B, N), np.float64)
    if B and N:
        rc = lib.oracle_lse_backward(arr.ctypes.data, DTYPE_CODES[dtype], B, N, row_stride,
                                     lse.ctypes.data, grad.ctypes.data, dx.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_lse_backward rejected its arguments")
    return dx


def _raw(x: np.ndarray, dtype: str) -> np.ndarray:
    """Contiguous raw-element view of ``x``: float32 for f32, 16-bit elements otherwise."""
    if dtype == "f32":
        if x.dtype != np.float32:
            raise TypeError("f32 oracle input must be a float32 array")
    elif x.dtype not in (np.uint16, np.float16, np.int16):
        raise TypeError(f"{dtype} oracle input must be 16-bit raw elements")
    return np.ascontiguousarray(x)


def _lse(lib, x: np.ndarray, dtype: str, B: int | None, N: int | None,
         row_stride: int | None) -> np.ndarray:
    """out[b] = log sum_n exp(x[b, n]) in float64.

    ``x`` is a 2-D array ``[B, row_stride]`` (only the first ``N`` columns are
    read), or a flat buffer with ``B``, ``N`` and ``row_stride`` given.  For
    bf16/f16 pass the raw 16-bit patterns (uint16) or float16 values.
    """
    if dtype not in DTYPE_CODES:
        raise ValueError(f"unknown dtype {dtype!r}")
    arr = _raw(x, dtype)
    if arr.ndim == 2:
        B = arr.shape[0] if B is None else B
        row_stride = arr.shape[1] if row_stride is None else row_stride
        N = row_stride if N is None else N
    elif B is None or N is None:
        raise ValueError("flat input needs B and N")
    row_stride = N if row_stride is None else row_stride
    if B > 0 and N > 0 and arr.size < (B - 1) * row_stride + N:
        raise ValueError("buffer smaller than (B-1)*row_stride + N elements")
    out = np.empty(max(B, 0), dtype=np.float64)
    rc = lib.oracle_lse(arr.ctypes.data if arr.size else None, DTYPE_CODES[dtype],
                        B, N, row_stride, out.ctypes.data if out.size else None)
    if rc != 0:
        raise ValueError(f"oracle_lse rejected B={B} N={N} row_stride={row_stride}")
    return out


def _decode(lib, x: np.ndarray, dtype: str) -> np.ndarray:
    arr = _raw(x, dtype).reshape(-1)
    out = np.empty(arr.size, dtype=np.float64)
    if arr.size:
        rc = lib.oracle_decode(arr.ctypes.data, DTYPE_CODES[dtype], arr.size,
                               out.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_decode failed")
    return out
