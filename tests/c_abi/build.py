"""Compile the C99 example caller against include/fa.h and libfa_gb300.so."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
LIBDIR = os.path.join(ROOT, "online_softmax_tiling_gb300")


def cuda_root() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def build(out_dir: str) -> str:
    exe = os.path.join(out_dir, "fa_example")
    cuda = cuda_root()
    libdirs = [os.path.join(cuda, d) for d in ("lib64", "lib", "targets/sbsa-linux/lib",
                                               "targets/x86_64-linux/lib")]
    libdirs = [d for d in libdirs if os.path.isdir(d)]
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(HERE, "fa_example.c"), "-o", exe,
           "-L", LIBDIR, "-lfa_gb300", "-Wl,-rpath," + LIBDIR]
    for d in libdirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lcudart"]
    subprocess.run(cmd, check=True)
    return exe
