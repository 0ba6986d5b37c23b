"""Build ``libfa.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m online_softmax_14_b300.build          # rebuild if stale
    python -m online_softmax_14_b300.build --force  # always rebuild

The library is one translation unit (``csrc/fa_lib.cu``, which includes the
kernel headers) linked against the static CUDA runtime; driver entry points
(``cuTensorMapEncodeTiled``) are resolved at run time, so the library needs no
GPU to build or to load.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libfa.so")
MAIN_SRC = os.path.join(PKG, "csrc", "fa_lib.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-v"]


def sources():
    return sorted(glob.glob(os.path.join(PKG, "csrc", "*.cu")) + glob.glob(os.path.join(PKG, "csrc", "*.cuh"))
                  + glob.glob(os.path.join(ROOT, "include", "*.h")))


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa.so if it is missing or older than a source; return its path."""
    if not force and not is_stale():
        return LIB
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, MAIN_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    log = r.stdout + r.stderr
    if "spill stores" in log:
        for line in log.splitlines():
            if "spill" in line and not line.strip().startswith("0 bytes stack frame, 0 bytes spill stores"):
                print("warning:", line.strip(), file=sys.stderr)
    if verbose:
        print(" ".join(cmd))
        print(log)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
