"""Loader of the CUDA twin of ``synth.gen`` (bit-identical device fills)."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_cuda.cu")
_LIB = os.path.join(_HERE, "libkamera_synth.so")
_lock = threading.Lock()
_lib = None

NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build_cmd(src: str = _SRC, out: str = _LIB) -> list[str]:
    return ["nvcc", *NVCC_ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-o", out, src]


def build() -> str:
    subprocess.run(build_cmd(), check=True)
    return _LIB


def load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build()
            lib = ctypes.CDLL(_LIB)
            i64, u64, f32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
            lib.synth_fill_rows.argtypes = [ctypes.c_void_p, i64, i64, i64, i64, i64, u64, u64, u64, u64, f32,
                                            u64, u64, u64, f32, ctypes.c_int32, ctypes.c_void_p]
            lib.synth_fill_rows.restype = ctypes.c_int
            _lib = lib
    return _lib


def fill_rows(out_ptr: int, *, n_slabs: int, rows: int, row_len: int, out_slab_stride: int, out_row_stride: int,
              stream: int, idx0: int, idx_slab_stride: int, idx_row_stride: int, scale: float,
              outlier_stream: int = 0, okey0: int = 0, okey_slab_stride: int = 0, outlier_scale: float = 0.0,
              outlier_permille: int = 0, cuda_stream: int = 0) -> None:
    lib = load()
    mask = (1 << 64) - 1
    rc = lib.synth_fill_rows(ctypes.c_void_p(out_ptr), n_slabs, rows, row_len, out_slab_stride, out_row_stride,
                             stream & mask, idx0 & mask, idx_slab_stride & mask, idx_row_stride & mask,
                             float(scale), outlier_stream & mask, okey0 & mask, okey_slab_stride & mask,
                             float(outlier_scale), int(outlier_permille), ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_rows: CUDA error {rc}")
