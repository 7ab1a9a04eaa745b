"""Build the CUDA library (libspecverify.so) in-tree for sm_103a.

    python -m draft_verification_02_b300.build [--force] [--verbose]

nvcc compiles csrc/*.cu for sm_103a only and links them into one shared
library next to this file, linked against the shared CUDA runtime (the same
libcudart the PyTorch process already has loaded).
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libspecverify.so")
# the bounds-checked build: every global index of the verification kernels is
# checked against its buffer (an out-of-range index sets the invalid-argument
# status bit and its access is skipped); the tests run parity cases on it
DEBUG_LIB = os.path.join(PKG, "libspecverify_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                     "-cudart", "shared", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(target: str, deps: list) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    """Compile csrc/*.cu into libspecverify.so (debug: libspecverify_debug.so,
    with -DSV_DEBUG) unless it is newer than every source."""
    lib = DEBUG_LIB if debug else LIB
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    if not force and not _stale(lib, deps):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    flags = [*(extra_flags or []), *(["-DSV_DEBUG"] if debug else [])]
    cmd = [nvcc(), *NVCC_FLAGS, *flags, "-o", tmp, *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the bounds-checked build")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose, debug=args.debug))


if __name__ == "__main__":
    main()
