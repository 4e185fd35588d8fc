"""Builds the CUDA library ``libflp.so`` in-tree with nvcc for sm_103a.

The library is one translation unit (``csrc/flp.cu``) that holds the C ABI of
``include/flp.h`` and the kernels.  Rebuilt when any source is newer than the
shared object.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libflp.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(PKG, "csrc", "*"))) + [os.path.join(ROOT, "include", "flp.h")]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libflp.so")
    return cand


def command(out: str, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-shared", "-I" + os.path.join(ROOT, "include"), "-o", out,
            os.path.join(PKG, "csrc", "flp.cu")] + (extra or [])


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if force or stale():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = command(tmp, ["-Xptxas", "-v"] if verbose else None)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
