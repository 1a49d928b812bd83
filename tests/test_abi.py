"""The C ABI without a GPU: the library loads, exports what include/lse.h
declares, lays out lse_plan as C does, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

import log_sum_exp_gb300 as L
from log_sum_exp_gb300 import build as lse_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lse.h")


@pytest.fixture(scope="module")
def lib():
    lse_build.build()
    return L.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^LSE_API\s+[\w\s\*]+?\b(lse_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_binding_names():
    assert declared_functions() == L.ABI_FUNCTIONS


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", L.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert {n for n in exported if n.startswith("lse_")} == set(declared_functions())


def test_plan_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "lse.h"\n'
                   'int main(void){printf("%zu", sizeof(lse_plan));'
                   + "".join(f'printf(" %zu", offsetof(lse_plan, {f}));'
                             for f, _ in L.LsePlan._fields_)
                   + "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), "-o", str(exe), str(src)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(L.LsePlan)] + [getattr(L.LsePlan, f).offset for f, _ in L.LsePlan._fields_]
    assert got == want


def test_status_strings(lib):
    for code, text in [(0, "ok"), (1, "invalid argument"), (2, "unsupported dtype"),
                       (3, "device scratch allocation failed"), (4, "CUDA error"),
                       (99, "unknown status")]:
        assert L.status_string(code) == text


@pytest.mark.parametrize("args,status", [
    ((16, 0, -1, 4, 4, 16), 1),            # B < 0
    ((16, 0, 4, -1, 4, 16), 1),            # N < 0
    ((16, 0, 4, 8, 7, 16), 1),             # row_stride < N
    ((0, 0, 4, 8, 8, 16), 1),              # x NULL with work to do
    ((16, 0, 4, 8, 8, 0), 1),              # out NULL
    ((16, 0, 4, 8, 8, 18), 1),             # out not 4-byte aligned
    ((18, 0, 4, 8, 8, 16), 1),             # f32 x not element aligned
    ((17, 1, 4, 8, 8, 16), 1),             # bf16 x not element aligned
    ((16, 3, 4, 8, 8, 16), 2),             # unknown dtype
    ((16, 0, 1 << 40, 1 << 30, 1 << 30, 16), 1),  # byte extent overflows int64
])
def test_bad_arguments_rejected_before_cuda(lib, args, status):
    x, dt, B, N, stride, out = args
    for fn in (lib.lse_forward, lib.lse_forward_host):
        assert fn(x or None, dt, B, N, stride, out or None, None) == status
    assert lib.lse_forward_plan(x or None, dt, B, N, stride, out or None, None, None, None,
                                None) == status


def test_zero_rows_is_ok_without_device(lib):
    assert lib.lse_forward(None, 0, 0, 5, 5, None, None) == 0


def test_last_cuda_error_null(lib):
    assert lib.lse_last_cuda_error(None) == 1
    v = ctypes.c_int(-1)
    assert lib.lse_last_cuda_error(ctypes.byref(v)) == 0


@pytest.mark.parametrize("args,status", [
    # x, dtype, A, R, C, sa, sr, lse, grad, dx, dsa, dsr
    ((16, 0, -1, 2, 4, 8, 4, 16, 16, 16, 8, 4), 1),     # A < 0
    ((16, 0, 2, 2, 4, -8, 4, 16, 16, 16, 8, 4), 1),     # negative stride
    ((16, 0, 2, 2, 4, 8, 4, 16, 16, 16, 8, -4), 1),     # negative dx stride
    ((0, 0, 2, 2, 4, 8, 4, 16, 16, 16, 8, 4), 1),       # x NULL with work to do
    ((16, 0, 2, 2, 4, 8, 4, 0, 16, 16, 8, 4), 1),       # lse NULL
    ((16, 0, 2, 2, 4, 8, 4, 16, 16, 0, 8, 4), 1),       # dx NULL
    ((16, 0, 2, 2, 4, 8, 4, 18, 16, 16, 8, 4), 1),      # lse not 4-byte aligned
    ((16, 1, 2, 2, 4, 8, 4, 16, 16, 17, 8, 4), 1),      # dx not element aligned
    ((16, 5, 2, 2, 4, 8, 4, 16, 16, 16, 8, 4), 2),      # unknown dtype
    ((16, 0, 2, 1 << 40, 4, 8, 1 << 30, 16, 16, 16, 8, 4), 1),  # x extent overflows
])
def test_backward_strided_bad_arguments_rejected_before_cuda(lib, args, status):
    x, dt, A, R, C, sa, sr, lse, grad, dx, dsa, dsr = args
    assert lib.lse_backward_strided(x or None, dt, A, R, C, sa, sr, lse or None, grad or None,
                                    dx or None, dsa, dsr, None) == status


def test_backward_strided_empty_is_ok_without_device(lib):
    assert lib.lse_backward_strided(None, 0, 0, 3, 4, 12, 4, None, None, None, 12, 4, None) == 0
    assert lib.lse_backward_strided(None, 0, 2, 0, 4, 0, 4, None, None, None, 0, 4, None) == 0


@pytest.mark.parametrize("dt,x", [(0, 18), (0, 17), (1, 17), (2, 33)])
def test_misaligned_x_rejected_before_cuda(lib, dt, x):
    """Every load is at least one whole element: an x that is not element
    aligned is refused by every entry point, before any device work."""
    B, N, out, t, lp = 4, 8, 256, 512, 1024
    assert lib.lse_forward(x, dt, B, N, N, out, None) == 1
    assert lib.lse_forward_host(x, dt, B, N, N, out, None) == 1
    assert lib.lse_forward_plan(x, dt, B, N, N, out, None, None, None, None) == 1
    assert lib.lse_forward16(x, dt, B, N, N, out, None, None) == 1
    assert lib.lse_forward_split_static(x, dt, B, N, N, out, None) == 1
    assert lib.lse_token_logprob(x, dt, B, N, N, t, lp, None, None) == 1
    assert lib.lse_backward(x, dt, B, N, N, out, out, 2048, N, None) == 1
    assert lib.lse_forward_strided(x, dt, 2, 3, N, 3 * N, N, out, None, None) == 1
    assert lib.lse_backward_strided(x, dt, 2, 3, N, 3 * N, N, out, out, 2048, 3 * N, N, None) == 1
