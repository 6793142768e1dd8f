"""Compile libhq.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

No fast-math: the kernels rely on IEEE division, correctly rounded reciprocals and
denormal support.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "hq.cu"), os.path.join(CSRC, "hq_host.cu"),
           os.path.join(CSRC, "hq_noalloc.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "hq_kernels.cuh"), os.path.join(CSRC, "hq_int8.cuh"),
                  os.path.join(CSRC, "hq_internal.h"),
                  os.path.join(INCLUDE, "hq.h")]
LIB = os.path.join(PKG, "libhq.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhq.so")


def nvcc_command(out: str, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
            "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, *(extra or []), "-o", out,
            *SOURCES]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else None)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
