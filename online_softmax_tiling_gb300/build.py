"""Build the sm_103a shared library in-tree with nvcc (no CMake, two translation units)."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("fa_api.cu", "ceilings.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("fa_fwd_kernel.cuh", "fa_fwd_qtile_kernel.cuh", "fa_fwd_wide_kernel.cuh",
                                                     "naive_attention.cuh",
                                                     "sm103_ptx.cuh")] + [
    os.path.join(ROOT, "include", f) for f in ("fa.h", "fa_ceilings.h", "fa_naive.h")]
LIBRARY = os.path.join(HERE, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise FileNotFoundError("nvcc not found (CUDA 13 toolkit required)")
    return cand


def stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(p) > t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa_gb300.so for sm_103a (static cudart, -O3 -lineinfo)."""
    if not force and not stale():
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "--threads", "2", "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose=True))
