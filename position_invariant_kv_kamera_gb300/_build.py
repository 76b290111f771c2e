"""Build of the in-tree CUDA library ``libkamera.so`` (sm_103a only)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkamera.so")
SOURCES = [os.path.join(CSRC, "kamera_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("kamera_kernel.cuh", "kamera_factor.cuh", "kamera_orbit.cuh", "kamera_compress.cuh", "ptx.cuh")] + [os.path.join(INCLUDE, "kamera.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-shared"]


def build_cmd(out: str = LIB, extra: list[str] | None = None) -> list[str]:
    return ["nvcc", *NVCC_FLAGS, *(extra or []), "-I" + INCLUDE, "-I" + CSRC, "-o", out, *SOURCES]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False) -> str:
    if force or stale():
        subprocess.run(build_cmd(), check=True)
    return LIB
