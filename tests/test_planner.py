"""The kernel-mapping rules on the CPU: tests/c/planner_check.cu compiles the
library's planner against a stand-in device description (152 SMs) and checks
the plans it makes for the workload shapes and the documented rules."""
import glob
import os
import subprocess

import pytest

from log_sum_exp_gb300 import build as lse_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_planner_rules(tmp_path):
    lse_build.build()
    objs = [o for o in glob.glob(os.path.join(lse_build.BUILD, "*.o"))
            if os.path.basename(o) != "lse_api.o"]
    if not objs:
        pytest.skip("library objects not built")
    exe = tmp_path / "planner_check"
    subprocess.run([lse_build._nvcc(), *lse_build.ARCH_FLAGS, "-O1", "-std=c++17",
                    "-I", lse_build.INCLUDE, "-o", str(exe),
                    os.path.join(ROOT, "tests", "c", "planner_check.cu"), *objs,
                    "-Xlinker", f"-rpath,{lse_build._cuda_lib_dir()}"],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "planner: ok" in r.stdout
