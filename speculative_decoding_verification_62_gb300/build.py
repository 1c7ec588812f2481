"""Compile the CUDA verify library (sm_103a) into the package directory.

One translation unit, one -gencode: nvcc cross-compiles here without a GPU
and builds natively on the GPU host in a few seconds.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libspec_verify.so")
SOURCES = [os.path.join(PKG, "csrc", "spec_verify.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA verify library cannot be built")
    return path


def inputs() -> list[str]:
    return SOURCES + glob.glob(os.path.join(PKG, "csrc", "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libspec_verify.so if it is missing or older than its sources."""
    if not (force or stale()):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-O3", *ARCH, "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I", INCLUDE, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
