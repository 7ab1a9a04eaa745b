"""Parity cases on the bounds-checked build (libspecverify_debug.so, compiled
with -DSV_DEBUG): every global index the verification kernels form is checked
against its buffer, and an out-of-range one sets the invalid-argument status
bit instead of being accessed.  The cases (the tiny configuration, the shape
sweep with ragged tails and unaligned rows, the padded draft layout, draws by
clusters of 4 CTAs at full depth, host row bounds far above the real rows)
must give the oracle's results with a clean device status, so no index left
its buffer.
Run in a child process so that the binding loads the debug library."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_parity_cases_on_the_bounds_checked_build():
    env = dict(os.environ, SPECVERIFY_LIB="libspecverify_debug.so")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_gpu_verify.py"),
         "-k", "tiny_config or shapes or padded_draft_layout or four_cta_draws or loose"],
        env=env, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "failed" not in r.stdout, r.stdout[-2000:]


@pytest.mark.gpu
def test_sharded_parity_cases_on_the_bounds_checked_build():
    """The vocabulary-sharded kernels on the same build: uneven shard widths
    (plain-load rows), the padded draft layout and a loose row bound."""
    env = dict(os.environ, SPECVERIFY_LIB="libspecverify_debug.so")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_gpu_shard.py"),
         "-k", "(matches_oracle and (4099 or 12345)) or padded_draft_layout or loose_row_bound"],
        env=env, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "failed" not in r.stdout, r.stdout[-2000:]
