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
import re
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


def spilling_kernels(ptxas_log: str) -> list:
    """Kernels for which ptxas -v reports spill stores or loads, with the line."""
    out, kernel = [], None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            kernel = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and (int(m.group(1)) or int(m.group(2))):
            out.append(f"{kernel}: {line.strip()}")
    return out


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
    spills = spilling_kernels(log)
    if spills:
        raise RuntimeError("register spills (every kernel must report 0 bytes):\n" + "\n".join(spills))
    if verbose:
        print(" ".join(cmd))
        print(log)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
