"""The streaming pass's unit planner (plan() in csrc/verify_params.cuh) on
the CPU: tests/plan_check.cu includes the header, is compiled with nvcc and
runs on the host (no kernel is launched).  It checks the split's invariants
over many shapes, that a short pass takes the largest unit, and the unit
sizes that the B300 measurements behind the rule chose."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "draft_verification_02_b300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "plan_check.cu")


def _nvcc():
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


@pytest.mark.skipif(_nvcc() is None, reason="needs nvcc")
def test_unit_planner(tmp_path):
    exe = str(tmp_path / "plan_check")
    subprocess.run([_nvcc(), "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-x", "cu", "-I", INCLUDE, "-I", CSRC, SRC, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "failures 0" in r.stdout, r.stdout
