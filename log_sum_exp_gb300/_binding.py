"""ctypes binding of liblse (include/lse.h).  Argument marshalling only.

Every function here passes pointers, sizes and the CUDA stream to the C ABI;
all arithmetic runs in liblse's kernels.  There is no CPU fallback: if the
library is missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LSE_OK = 0
STATUS_NAMES = {0: "LSE_OK", 1: "LSE_ERR_INVALID_ARG", 2: "LSE_ERR_UNSUPPORTED_DTYPE",
                3: "LSE_ERR_ALLOC", 4: "LSE_ERR_CUDA"}
DTYPES = {"f32": 0, "bf16": 1, "f16": 2}
PATHS = {"auto": 0, "empty": 1, "subwarp": 2, "cta": 3, "split": 4, "columns_warp": 5,
         "columns_cta": 6, "rowtile": 7, "columns_short": 8}
PATH_NAMES = {v: k for k, v in PATHS.items()}

# Exported names, in header order.
ABI_FUNCTIONS = ["lse_forward", "lse_plan_query", "lse_forward_plan", "lse_forward16",
                 "lse_forward_host", "lse_token_logprob", "lse_token_logprob_plan",
                 "lse_backward", "lse_forward_strided", "lse_backward_strided",
                 "lse_trim_memory", "lse_wait_timeouts", "lse_set_wait_limit", "lse_status_string",
                 "lse_last_cuda_error", "lse_forward_split_static"]


class LsePlan(ctypes.Structure):
    """Mirror of ``lse_plan``."""
    _fields_ = [
        ("path", ctypes.c_int32),
        ("vector_bytes", ctypes.c_int32),
        ("lanes_per_row", ctypes.c_int32),
        ("slots_per_lane", ctypes.c_int32),
        ("threads", ctypes.c_int32),
        ("launches", ctypes.c_int32),
        ("splits", ctypes.c_int64),
        ("segment_slots", ctypes.c_int64),
        ("grid", ctypes.c_int64),
        ("scratch_bytes", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["path"] = PATH_NAMES.get(self.path, self.path)
        return d


class LseError(RuntimeError):
    def __init__(self, status: int, where: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        if cuda_error:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load liblse.so; raise if it has not been built."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"liblse.so is not built ({path}); run "
                              "log_sum_exp_gb300.build.build() first")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.lse_forward.argtypes = [vp, i32, i64, i64, i64, vp, vp]
        lib.lse_forward.restype = i32
        lib.lse_plan_query.argtypes = [vp, i32, i64, i64, i64, ctypes.POINTER(LsePlan)]
        lib.lse_plan_query.restype = i32
        lib.lse_forward_plan.argtypes = [vp, i32, i64, i64, i64, vp, vp,
                                         ctypes.POINTER(LsePlan), vp, vp]
        lib.lse_forward_plan.restype = i32
        lib.lse_forward16.argtypes = [vp, i32, i64, i64, i64, vp, vp, ctypes.POINTER(LsePlan)]
        lib.lse_forward16.restype = i32
        lib.lse_forward_host.argtypes = [vp, i32, i64, i64, i64, vp, vp]
        lib.lse_forward_host.restype = i32
        lib.lse_token_logprob.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp, vp]
        lib.lse_token_logprob.restype = i32
        lib.lse_token_logprob_plan.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp, vp,
                                               ctypes.POINTER(LsePlan)]
        lib.lse_token_logprob_plan.restype = i32
        lib.lse_backward.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp, i64, vp]
        lib.lse_backward.restype = i32
        lib.lse_forward_strided.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp, vp,
                                            ctypes.POINTER(LsePlan)]
        lib.lse_forward_strided.restype = i32
        lib.lse_backward_strided.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp, vp, vp, i64,
                                             i64, vp]
        lib.lse_backward_strided.restype = i32
        lib.lse_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
        lib.lse_wait_timeouts.restype = i32
        lib.lse_set_wait_limit.argtypes = [ctypes.c_uint32]
        lib.lse_set_wait_limit.restype = i32
        lib.lse_trim_memory.argtypes = []
        lib.lse_trim_memory.restype = i32
        lib.lse_status_string.argtypes = [i32]
        lib.lse_status_string.restype = ctypes.c_char_p
        lib.lse_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.lse_last_cuda_error.restype = i32
        _lib = lib
        return lib


def _check(status: int, where: str) -> None:
    if status != LSE_OK:
        err = ctypes.c_int(0)
        load().lse_last_cuda_error(ctypes.byref(err))
        raise LseError(status, where, err.value)


def lse_trim_memory() -> None:
    """Release the library's cached device memory on the current device."""
    _check(load().lse_trim_memory(), "lse_trim_memory")


def lse_wait_timeouts() -> int:
    """Bounded device-side waits that gave up so far (0 in correct operation)."""
    v = ctypes.c_ulonglong(0)
    _check(load().lse_wait_timeouts(ctypes.byref(v)), "lse_wait_timeouts")
    return v.value


DEFAULT_WAIT_POLLS = 1 << 26


def lse_set_wait_limit(polls: int) -> None:
    """Testing aid: poll limit of the bulk-copy ring's stage waits for later
    launches (DEFAULT_WAIT_POLLS restores it; 0 gives up at once)."""
    _check(load().lse_set_wait_limit(polls), "lse_set_wait_limit")


def status_string(status: int) -> str:
    return load().lse_status_string(status).decode()


# ---------------------------------------------------------------------------
# Raw-pointer calls (same names and argument order as the C ABI).
# ---------------------------------------------------------------------------
def lse_forward_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int, out_ptr: int,
                    stream: int = 0) -> None:
    _check(load().lse_forward(x_ptr or None, DTYPES[dtype], B, N, row_stride, out_ptr or None,
                              stream or None), "lse_forward")


def lse_forward_plan_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int, out_ptr: int,
                         stream: int = 0, plan: LsePlan | None = None, ev_begin: int = 0,
                         ev_end: int = 0) -> LsePlan:
    p = plan if plan is not None else LsePlan()
    _check(load().lse_forward_plan(x_ptr or None, DTYPES[dtype], B, N, row_stride, out_ptr or None,
                                   stream or None, ctypes.byref(p), ev_begin or None,
                                   ev_end or None), "lse_forward_plan")
    return p


def lse_forward16_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int, out_ptr: int,
                      stream: int = 0, plan: LsePlan | None = None) -> LsePlan:
    p = plan if plan is not None else LsePlan()
    _check(load().lse_forward16(x_ptr or None, DTYPES[dtype], B, N, row_stride, out_ptr or None,
                                stream or None, ctypes.byref(p)), "lse_forward16")
    return p


def lse_plan_query_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int) -> LsePlan:
    p = LsePlan()
    _check(load().lse_plan_query(x_ptr or None, DTYPES[dtype], B, N, row_stride, ctypes.byref(p)),
           "lse_plan_query")
    return p


def lse_forward_host_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int, out_ptr: int,
                         stream: int = 0) -> None:
    _check(load().lse_forward_host(x_ptr or None, DTYPES[dtype], B, N, row_stride, out_ptr or None,
                                   stream or None), "lse_forward_host")


def lse_token_logprob_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int,
                          target_ptr: int, logprob_ptr: int, lse_ptr: int = 0, stream: int = 0,
                          plan: LsePlan | None = None) -> LsePlan:
    p = plan if plan is not None else LsePlan()
    _check(load().lse_token_logprob_plan(x_ptr or None, DTYPES[dtype], B, N, row_stride,
                                         target_ptr or None, logprob_ptr or None, lse_ptr or None,
                                         stream or None, ctypes.byref(p)), "lse_token_logprob")
    return p


def lse_backward_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int, lse_ptr: int,
                     grad_ptr: int, dx_ptr: int, dx_row_stride: int, stream: int = 0) -> None:
    _check(load().lse_backward(x_ptr or None, DTYPES[dtype], B, N, row_stride, lse_ptr or None,
                               grad_ptr or None, dx_ptr or None, dx_row_stride, stream or None),
           "lse_backward")


def lse_forward_strided_ptr(x_ptr: int, dtype: str, A: int, R: int, C: int, stride_a: int,
                            stride_r: int, out_ptr: int, stream: int = 0,
                            plan: LsePlan | dict | None = None) -> LsePlan:
    p = _as_plan(plan) if plan is not None else LsePlan()
    _check(load().lse_forward_strided(x_ptr or None, DTYPES[dtype], A, R, C, stride_a, stride_r,
                                      out_ptr or None, stream or None, ctypes.byref(p)),
           "lse_forward_strided")
    return p


def lse_backward_strided_ptr(x_ptr: int, dtype: str, A: int, R: int, C: int, stride_a: int,
                             stride_r: int, lse_ptr: int, grad_ptr: int, dx_ptr: int,
                             dx_stride_a: int, dx_stride_r: int, stream: int = 0) -> None:
    _check(load().lse_backward_strided(x_ptr or None, DTYPES[dtype], A, R, C, stride_a, stride_r,
                                       lse_ptr or None, grad_ptr or None, dx_ptr or None,
                                       dx_stride_a, dx_stride_r, stream or None),
           "lse_backward_strided")


def lse_forward_split_static_ptr(x_ptr: int, dtype: str, B: int, N: int, row_stride: int,
                                 out_ptr: int, stream: int = 0) -> None:
    """The split-row mapping with no device allocation (fixed 1 MiB scratch).

    For callers that may not allocate device memory during the call.  Calls
    whose kernels overlap on the GPU share the scratch and must not run
    concurrently; make the first call on a device before any stream capture.
    """
    fn = load().lse_forward_split_static
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, i32, i64, i64, i64, vp, vp]
    fn.restype = i32
    _check(fn(x_ptr or None, DTYPES[dtype], B, N, row_stride, out_ptr or None, stream or None),
           "lse_forward_split_static")


# ---------------------------------------------------------------------------
# torch-tensor conveniences: torch supplies device memory and the stream only.
# ---------------------------------------------------------------------------
_TORCH = None
_DTYPE_NAMES = None


def _torch():
    global _TORCH
    if _TORCH is None:
        import torch
        _TORCH = torch
    return _TORCH


def _dtype_name(t) -> str:
    global _DTYPE_NAMES
    if _DTYPE_NAMES is None:
        torch = _torch()
        _DTYPE_NAMES = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
    name = _DTYPE_NAMES.get(t.dtype)
    if name is None:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float32, bfloat16 or float16")
    return name


class _on_device:
    """Make ``device`` current for the block, switching only when it is not
    current already (torch.cuda.device always switches)."""

    __slots__ = ("index", "prev")

    def __init__(self, device):
        self.index = device.index

    def __enter__(self):
        cuda = _torch().cuda
        cur = cuda.current_device()
        self.prev = cur if self.index is not None and cur != self.index else None
        if self.prev is not None:
            cuda.set_device(self.index)

    def __exit__(self, *exc):
        if self.prev is not None:
            _torch().cuda.set_device(self.prev)


def _rows(x):
    """(B, N, row_stride) of a 1-D or 2-D tensor whose last dimension has unit stride."""
    if x.dim() == 1:
        if x.numel() > 1 and x.stride(0) != 1:
            raise ValueError("the reduced dimension must have unit stride")
        return 1, x.shape[0], x.shape[0]
    if x.dim() != 2:
        raise ValueError("expected a [B, N] tensor (reduce over the last dimension)")
    B, N = x.shape
    if N > 1 and x.stride(1) != 1:
        raise ValueError("the reduced (last) dimension must have unit stride")
    row_stride = x.stride(0) if B > 1 else N
    if row_stride < N:
        raise ValueError("rows overlap (row stride < N)")
    return B, N, row_stride


_RAW_STREAM = None


def _stream_handle(stream, device):
    """cudaStream_t of ``stream``, or of the device's current stream.  The raw
    getter avoids building a torch Stream object on every call."""
    global _RAW_STREAM
    if stream is not None:
        return stream.cuda_stream
    torch = _torch()
    if _RAW_STREAM is None:
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    index = device.index if device.index is not None else torch.cuda.current_device()
    if _RAW_STREAM:
        return _RAW_STREAM(index)
    return torch.cuda.current_stream(index).cuda_stream


def lse_forward(x, out=None, stream=None):
    """out[b] = log sum_n exp(x[b, n]) for a CUDA tensor x of shape [B, N] (or [N]).

    Returns a float32 tensor of shape [B] (a 0-d tensor for 1-D input).
    """
    torch = _torch()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (use lse_forward_host for host memory)")
    dt = _dtype_name(x)
    B, N, row_stride = _rows(x)
    out = _out_rows(out, B, x)
    device = x.device
    args = (x.data_ptr() or None, DTYPES[dt], B, N, row_stride, out.data_ptr() or None,
            _stream_handle(stream, device) or None)
    if torch.cuda.current_device() == device.index:
        _check(load().lse_forward(*args), "lse_forward")
    else:
        with _on_device(device):
            _check(load().lse_forward(*args), "lse_forward")
    return out.reshape(()) if x.dim() == 1 else out


def _out_rows(out, B, x):
    """A float32 [B] output on x's device: new, or the caller's after checks."""
    torch = _torch()
    if out is None:
        return torch.empty(B, dtype=torch.float32, device=x.device)
    if out.dtype != torch.float32 or out.numel() != B or not out.is_contiguous() \
            or out.device != x.device:
        raise ValueError("out must be a contiguous float32 tensor of B elements on x's device")
    return out


def lse_forward_plan(x, plan: LsePlan | dict | None = None, out=None, stream=None,
                     ev_begin=None, ev_end=None):
    """``lse_forward`` with an optional forced plan and timing events.

    ``plan`` may be an LsePlan or a dict of its fields (``path`` may be a name).
    ``ev_begin``/``ev_end`` are torch.cuda.Event objects recorded around the
    main kernel.  Returns (out, plan_that_ran).
    """
    torch = _torch()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (use lse_forward_host for host memory)")
    dt = _dtype_name(x)
    B, N, row_stride = _rows(x)
    if out is None:
        out = torch.empty(B, dtype=torch.float32, device=x.device)
    elif out.dtype != torch.float32 or out.numel() != B or not out.is_contiguous() \
            or out.device != x.device:
        raise ValueError("out must be a contiguous float32 tensor of B elements on x's device")
    p = _as_plan(plan)
    with _on_device(x.device):
        evb = _event_handle(ev_begin)
        eve = _event_handle(ev_end)
        p = lse_forward_plan_ptr(x.data_ptr(), dt, B, N, row_stride, out.data_ptr(),
                                 _stream_handle(stream, x.device), p, evb, eve)
    if x.dim() == 1:
        return out.reshape(()), p
    return out, p


def lse_forward16(x, plan: LsePlan | dict | None = None, out=None, stream=None):
    """``lse_forward`` with reduced-bit exponentials (two terms per packed bf16
    SFU operation; f32 sums).  Returns (out, plan_that_ran)."""
    torch = _torch()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    dt = _dtype_name(x)
    B, N, row_stride = _rows(x)
    if out is None:
        out = torch.empty(B, dtype=torch.float32, device=x.device)
    elif out.dtype != torch.float32 or out.numel() != B or not out.is_contiguous() \
            or out.device != x.device:
        raise ValueError("out must be a contiguous float32 tensor of B elements on x's device")
    p = _as_plan(plan)
    with _on_device(x.device):
        p = lse_forward16_ptr(x.data_ptr(), dt, B, N, row_stride, out.data_ptr(),
                              _stream_handle(stream, x.device), p)
    if x.dim() == 1:
        return out.reshape(()), p
    return out, p


def _event_handle(ev) -> int:
    if ev is None:
        return 0
    if isinstance(ev, int):
        return ev
    if ev.cuda_event == 0:  # torch creates the event lazily on first record
        ev.record()
    return ev.cuda_event


def _as_plan(plan) -> LsePlan | None:
    if plan is None or isinstance(plan, LsePlan):
        return plan
    p = LsePlan()
    for k, v in plan.items():
        if k == "path" and isinstance(v, str):
            v = PATHS[v]
        setattr(p, k, v)
    return p


def lse_token_logprob(x, target, lse_out=None, plan=None, stream=None, return_plan=False):
    """logprob[b] = x[b, target[b]] - logsumexp(x[b, :]) for a CUDA [B, N] tensor.

    ``target`` is a CUDA int64 tensor of B column indices (out-of-range -> NaN).
    ``lse_out`` (optional float32 [B]) receives the row values.  Returns the
    float32 [B] log-probabilities (and the plan that ran if ``return_plan``).
    """
    torch = _torch()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    dt = _dtype_name(x)
    B, N, row_stride = _rows(x)
    if target.dtype != torch.int64 or target.device != x.device or target.numel() != B \
            or not target.is_contiguous():
        raise ValueError("target must be a contiguous int64 tensor of B elements on x's device")
    logprob = torch.empty(B, dtype=torch.float32, device=x.device)
    if lse_out is not None and (lse_out.dtype != torch.float32 or lse_out.numel() != B
                                or not lse_out.is_contiguous() or lse_out.device != x.device):
        raise ValueError("lse_out must be a contiguous float32 tensor of B elements on x's device")
    with _on_device(x.device):
        p = lse_token_logprob_ptr(x.data_ptr(), dt, B, N, row_stride, target.data_ptr(),
                                  logprob.data_ptr(), lse_out.data_ptr() if lse_out is not None else 0,
                                  _stream_handle(stream, x.device), _as_plan(plan))
    return (logprob, p) if return_plan else logprob


def lse_backward(x, lse, grad, dx=None, stream=None):
    """dx[b, n] = grad[b] * exp(x[b, n] - lse[b]) for a CUDA [B, N] tensor x.

    ``lse`` and ``grad`` are float32 CUDA tensors of B elements; ``dx`` (optional)
    has x's dtype and shape.  Returns dx.
    """
    torch = _torch()
    dt = _dtype_name(x)
    B, N, row_stride = _rows(x)
    for name, t in (("lse", lse), ("grad", grad)):
        if t.dtype != torch.float32 or t.numel() != B or not t.is_contiguous() \
                or t.device != x.device:
            raise ValueError(f"{name} must be a contiguous float32 tensor of B elements")
    if dx is None:
        dx = torch.empty((B, N), dtype=x.dtype, device=x.device)
    if dx.shape != (B, N) or dx.dtype != x.dtype or (N > 1 and dx.stride(1) != 1):
        raise ValueError("dx must match x's shape and dtype with unit last stride")
    dx_stride = dx.stride(0) if B > 1 else N
    with _on_device(x.device):
        lse_backward_ptr(x.data_ptr(), dt, B, N, row_stride, lse.data_ptr(), grad.data_ptr(),
                         dx.data_ptr(), dx_stride, _stream_handle(stream, x.device))
    return dx


def logsumexp(x, dim=-1, keepdim=False, stream=None):
    """torch.logsumexp(x, dim, keepdim) on liblse for CUDA tensors, computed in f32.

    The reduced dimension may be any dimension; the tensor must be contiguous
    (its other dimensions collapse to (outer, inner)).  Returns float32 with
    ``dim`` removed.  When x requires a gradient the result is differentiable:
    the gradient g * exp(x - lse) comes from lse_backward (last dimension) or
    lse_backward_strided (any other).
    """
    torch = _torch()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if x.dim() == 0:
        raise ValueError("x must have at least one dimension")
    d = dim % x.dim()
    if torch.is_grad_enabled() and x.requires_grad:
        return _logsumexp_function().apply(x, d, keepdim, stream)
    return _logsumexp_value(x, d, keepdim, stream)


def _logsumexp_value(x, d, keepdim, stream):
    torch = _torch()
    dt = _dtype_name(x)
    shape = list(x.shape)
    R = shape[d]
    outer = 1
    for n in shape[:d]:
        outer *= n
    inner = 1
    for n in shape[d + 1:]:
        inner *= n
    out_shape = shape[:d] + shape[d + 1:]
    if not x.is_contiguous():
        raise ValueError("logsumexp needs a contiguous tensor")
    device = x.device
    out = torch.empty(out_shape, dtype=torch.float32, device=device)
    h = _stream_handle(stream, device)
    with _on_device(device):
        if inner == 1:
            lse_forward_ptr(x.data_ptr(), dt, outer, R, R, out.data_ptr(), h)
        else:
            lse_forward_strided_ptr(x.data_ptr(), dt, outer, R, inner, R * inner, inner,
                                    out.data_ptr(), h)
    return out.unsqueeze(d) if keepdim else out


_LSE_FUNCTION = None


def _logsumexp_function():
    """The torch.autograd.Function behind a differentiable logsumexp (built on
    first use, since torch is imported lazily)."""
    global _LSE_FUNCTION
    if _LSE_FUNCTION is None:
        torch = _torch()

        class LogSumExp(torch.autograd.Function):
            @staticmethod
            def forward(ctx, x, d, keepdim, stream):
                out = _logsumexp_value(x, d, keepdim, stream)
                ctx.save_for_backward(x, out)
                ctx.d, ctx.stream = d, stream
                return out

            @staticmethod
            def backward(ctx, grad_out):
                x, out = ctx.saved_tensors
                d = ctx.d
                R = x.shape[d]
                inner = 1
                for n in x.shape[d + 1:]:
                    inner *= n
                outer = x.numel() // (R * inner) if R * inner else 0
                g = grad_out.reshape(outer * inner).to(torch.float32).contiguous()
                lse = out.reshape(outer * inner)
                if inner == 1:
                    dx = lse_backward(x.reshape(outer, R), lse, g, stream=ctx.stream)
                    return dx.reshape(x.shape), None, None, None
                dx = torch.empty_like(x)
                with _on_device(x.device):
                    lse_backward_strided_ptr(x.data_ptr(), _dtype_name(x), outer, R, inner,
                                             R * inner, inner, lse.data_ptr(), g.data_ptr(),
                                             dx.data_ptr(), R * inner, inner,
                                             _stream_handle(ctx.stream, x.device))
                return dx, None, None, None

        _LSE_FUNCTION = LogSumExp
    return _LSE_FUNCTION


def lse_plan_query(x=None, dtype: str | None = None, B: int | None = None, N: int | None = None,
                   row_stride: int | None = None) -> dict:
    """The plan lse_forward would use, for a tensor or for (dtype, B, N, row_stride)."""
    if x is not None:
        dtype = _dtype_name(x)
        B, N, row_stride = _rows(x)
        ptr = x.data_ptr()
    else:
        ptr = 0
        row_stride = N if row_stride is None else row_stride
    return lse_plan_query_ptr(ptr, dtype, B, N, row_stride).as_dict()


def lse_forward_host(x, stream=None):
    """lse over a HOST tensor: the result for x in host memory, synchronised.

    ``x`` is a CPU torch tensor of shape [B, N].  A pinned ``x`` is streamed by
    the kernel in place (zero copy); a pageable one is copied to the device
    first.  Returns a CPU float32 tensor of shape [B] (pinned when x is).
    """
    torch = _torch()
    if x.is_cuda:
        raise ValueError("lse_forward_host takes host memory")
    dt = _dtype_name(x)
    B, N, row_stride = _rows(x)
    out = torch.empty(B, dtype=torch.float32, pin_memory=x.is_pinned())
    dev = torch.device("cuda", torch.cuda.current_device())
    lse_forward_host_ptr(x.data_ptr(), dt, B, N, row_stride, out.data_ptr(),
                         _stream_handle(stream, dev))
    return out
