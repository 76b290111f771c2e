"""Build of the in-tree CUDA library ``libkamera.so`` (sm_103a only).

Three translation units -- the host side with the reuse, encoder and orbit
kernels, and the two patch-formation kernel instances (the slowest code to
compile) -- are compiled in parallel, then linked into one shared library.
"""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkamera.so")
OBJDIR = os.path.join(PKG, "_build")
SOURCES = [os.path.join(CSRC, f) for f in ("kamera_api.cu", "kamera_factor_aligned.cu", "kamera_factor_general.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("kamera_kernel.cuh", "kamera_factor.cuh", "kamera_factor_launch.h",
                                            "kamera_orbit.cuh", "kamera_compress.cuh", "ptx.cuh")]
DEPS = SOURCES + HEADERS + [os.path.join(INCLUDE, "kamera.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC"]


def object_path(src: str, objdir: str = OBJDIR) -> str:
    return os.path.join(objdir, os.path.splitext(os.path.basename(src))[0] + ".o")


def compile_cmd(src: str, obj: str | None = None, extra: list[str] | None = None) -> list[str]:
    return ["nvcc", *NVCC_FLAGS, *(extra or []), "-I" + INCLUDE, "-I" + CSRC, "-c", "-o", obj or object_path(src),
            src]


def link_cmd(out: str = LIB, objs: list[str] | None = None) -> list[str]:
    return ["nvcc", *ARCH, "-shared", "-o", out, *(objs or [object_path(s) for s in SOURCES])]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, out: str = LIB, objdir: str = OBJDIR, extra: list[str] | None = None) -> str:
    """Compile the units in parallel and link them (only when a source is newer
    than the library, unless forced)."""
    if force or out != LIB or stale():
        os.makedirs(objdir, exist_ok=True)
        objs = [object_path(s, objdir) for s in SOURCES]
        procs = [subprocess.Popen(compile_cmd(s, o, extra)) for s, o in zip(SOURCES, objs)]
        failed = [(p.args, rc) for p in procs for rc in [p.wait()] if rc != 0]
        if failed:
            raise subprocess.CalledProcessError(failed[0][1], failed[0][0])
        subprocess.run(link_cmd(out, objs), check=True)
    return out
