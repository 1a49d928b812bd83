"""liblse from plain C (tests/c/abi_smoke.c, compiled with gcc against
include/lse.h and the CUDA runtime): lse_forward and lse_forward16 results
checked against the oracle."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from lse_testutil import compare, compare_e16, e16_bound

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import log_sum_exp_gb300 as L  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_sum_exp_gb300 import build as lse_build
    lib = lse_build.build()
    out = tmp_path_factory.mktemp("c") / "abi_smoke"
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    subprocess.run(["gcc", "-std=c11", "-O2", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c", "abi_smoke.c"),
                    "-o", str(out), lib, "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{cuda}/lib64"], check=True)
    return str(out)


@pytest.mark.parametrize("dt,B,N", [(0, 64, 4096), (0, 1000, 32), (1, 33, 32000), (2, 7, 100003),
                                    (0, 3, 1 << 20)])
def test_c_program(exe, tmp_path, dt, B, N):
    xfile = tmp_path / "x.bin"
    res = subprocess.run([exe, str(dt), str(B), str(N), "7", str(xfile)], capture_output=True,
                         text=True, check=True)
    vals = np.array([[float(v) for v in ln.split()] for ln in res.stdout.splitlines()])
    dtype = ["f32", "bf16", "f16"][dt]
    raw = np.fromfile(xfile, dtype=np.float32 if dt == 0 else np.uint16).reshape(B, N)
    want = oracle.lse(raw, dtype)
    compare(vals[:, 0], want)
    compare_e16(vals[:, 1], want, e16_bound(raw, dtype, want))
