"""The integer forms of the cost-unit D-cut's binary64 operations
(csrc/fp64_exact.cuh) against the host's IEEE arithmetic, on the CPU: the
header is compiled for the host with g++ and run on random operands and
constructed ties.  The GPU tests then compare the kernel's depths and
benefits with the oracle bit for bit."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "draft_verification_02_b300", "csrc")
SRC = os.path.join(ROOT, "tests", "fp64_exact_check.cpp")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_integer_forms_round_like_ieee_binary64(tmp_path):
    exe = str(tmp_path / "fp64_exact_check")
    # -ffp-contract=off: the reference arithmetic must not be fused either
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-I", CSRC, SRC, "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
