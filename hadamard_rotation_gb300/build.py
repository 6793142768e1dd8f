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
SOURCES = [os.path.join(CSRC, "hq.cu"), os.path.join(CSRC, "hq_int8.cu"),
           os.path.join(CSRC, "hq_host.cu"), os.path.join(CSRC, "hq_noalloc.cu")]
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


def nvcc_compile_command(src: str, obj: str, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-c",
            "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, *(extra or []), "-o", obj, src]


def nvcc_link_command(objs: list[str], out: str) -> list[str]:
    return [nvcc_path(), ARCH, "-shared", "-o", out, *objs]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(CSRC, os.path.basename(src)[:-3] + tag + ".o") for src in SOURCES]
    extra = ["-Xptxas", "-v"] if verbose else None
    try:
        # one nvcc per translation unit, in parallel, then one link
        procs = [subprocess.Popen(nvcc_compile_command(src, obj, extra))
                 for src, obj in zip(SOURCES, objs)]
        rcs = [pr.wait() for pr in procs]
        for src, rc in zip(SOURCES, rcs):
            if rc != 0:
                raise subprocess.CalledProcessError(rc, f"nvcc -c {os.path.basename(src)}")
        tmp = LIB + tag
        subprocess.run(nvcc_link_command(objs, tmp), check=True)
        os.replace(tmp, LIB)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
