"""Build libwgrad.so (sm_103a) in-tree with nvcc.

    python -m implicit_gemm_gb300.build [--force]

The library lands in implicit_gemm_gb300/_lib/libwgrad.so (git-ignored).  It is
compiled for exactly one target, sm_103a; there is no other code path.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libwgrad.so")
SOURCES = [os.path.join(CSRC, "wgrad.cu"), os.path.join(CSRC, "plan.cpp")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "k_igemm.cuh", "k_depthwise.cuh", "k_dgrad.cuh", "plan.h")] + [
    os.path.join(ROOT, "include", "wgrad.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwgrad.so")


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    with _lock:
        if not force and not stale():
            return LIB
        os.makedirs(LIBDIR, exist_ok=True)
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), ARCH, "-lineinfo", "-O3", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
               "-Xcompiler", "-fvisibility=hidden", "-shared", "-I", os.path.join(ROOT, "include"), "-o", tmp,
               *SOURCES]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
