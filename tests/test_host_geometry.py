"""Host logic of the launch geometry, on the CPU: each check includes the
header that holds the logic, is compiled with nvcc and runs on the host (no
kernel is launched).
- tests/plan_check.cu: the streaming pass's unit planner (plan() in
  csrc/verify_params.cuh): the split's invariants over many shapes, a short
  pass takes the largest unit, and the unit sizes the B300 measurements
  behind the rule chose.
- tests/draw_geometry_check.cu: the final draw's cluster geometry
  (draw_geometry() in csrc/finish_kernel.cuh): 16, 8 or 4 CTAs per draw by
  batch size, one wave up to the SM count, the merge capacity at the largest
  depth, the slice table, and a geometry for every accepted vocabulary."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "draft_verification_02_b300", "csrc")
INCLUDE = os.path.join(ROOT, "include")


def _nvcc():
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def _run_check(tmp_path, name):
    exe = str(tmp_path / name)
    subprocess.run([_nvcc(), "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-x", "cu", "-I", INCLUDE, "-I", CSRC,
                    os.path.join(ROOT, "tests", name + ".cu"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "failures 0" in r.stdout, r.stdout


@pytest.mark.skipif(_nvcc() is None, reason="needs nvcc")
def test_unit_planner(tmp_path):
    _run_check(tmp_path, "plan_check")


@pytest.mark.skipif(_nvcc() is None, reason="needs nvcc")
def test_draw_geometry(tmp_path):
    _run_check(tmp_path, "draw_geometry_check")
