"""Python binding of the GB300 Kamera KV-reuse library (``libkamera.so``).

Argument marshalling only: every step of the operation runs in the CUDA
kernels behind the C ABI of ``include/kamera.h``.  The functions keep the C
names.  There is no fallback: if the library is missing, importing the
binding's functions raises.

Kamera (gist.science summary of "Kamera: Unified Position-Invariant
Multimodal KV Cache for Training-Free Reuse"), §2 reuse equation
KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

KAMERA_OK, KAMERA_ERR_NULL, KAMERA_ERR_INVALID_ARG, KAMERA_ERR_UNSUPPORTED, KAMERA_ERR_ALIGNMENT, KAMERA_ERR_CUDA = range(6)
KAMERA_MHA, KAMERA_GQA, KAMERA_MLA = 0, 1, 2
KAMERA_ROTATE_HALF, KAMERA_INTERLEAVED = 0, 1
KAMERA_PATCH_AFTER_ROTATION, KAMERA_PATCH_CANONICAL_FRAME = 0, 1
KAMERA_EFLAG_CHUNK_OOB, KAMERA_EFLAG_PAGE_OOB, KAMERA_EFLAG_PATCH_OOB, KAMERA_EFLAG_LEN, KAMERA_EFLAG_TIMEOUT = (
    1, 2, 4, 8, 16)

EXPORTS = ("kamera_reuse_batched", "kamera_relocate", "kamera_apply_patch", "kamera_factor_workspace_size",
           "kamera_factor_patches", "kamera_factor_patches_noalloc", "kamera_orbit_mean", "kamera_v_codebook",
           "kamera_compress_chunks", "kamera_reuse_compressed", "kamera_set_launch_tuning",
           "kamera_get_launch_tuning", "kamera_status_string", "kamera_last_error", "kamera_abi_version")
FACTOR_STATIC_SCRATCH_BYTES = 16 << 20


class kamera_model_desc(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int32), ("num_layers", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32), ("latent_dim", ctypes.c_int32),
                ("pairing", ctypes.c_int32), ("patch_frame", ctypes.c_int32), ("rope_base", ctypes.c_double),
                ("inv_freq", ctypes.c_void_p), ("rope_sections", ctypes.c_int32 * 3), ("reserved0", ctypes.c_int32),
                ("section_delta", ctypes.c_void_p)]


class kamera_chunk_store(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("n_elems", ctypes.c_int64), ("offset", ctypes.c_void_p),
                ("len", ctypes.c_void_p), ("n_chunks", ctypes.c_int32)]


class kamera_patch_store(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("n_elems", ctypes.c_int64), ("offset", ctypes.c_void_p),
                ("len", ctypes.c_void_p), ("n_patches", ctypes.c_int32), ("rank", ctypes.c_int32)]


class kamera_paged_pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_size", ctypes.c_int32), ("block_table", ctypes.c_void_p), ("n_seqs", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32)]


class kamera_factor_desc(ctypes.Structure):
    _fields_ = [("delta", ctypes.c_void_p), ("delta_stride", ctypes.c_int64), ("n_slabs", ctypes.c_int32),
                ("T", ctypes.c_int32), ("D", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("oversample", ctypes.c_int32), ("power_iters", ctypes.c_int32), ("omega", ctypes.c_void_p)]


class kamera_compressed_store(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_norm", ctypes.c_void_p), ("row_offset", ctypes.c_void_p), ("len", ctypes.c_void_p),
                ("n_chunks", ctypes.c_int32), ("reserved", ctypes.c_int32), ("n_rows", ctypes.c_int64)]


class kamera_launch_tuning(ctypes.Structure):
    _fields_ = [("bn", ctypes.c_int32), ("stages", ctypes.c_int32), ("uv_slots", ctypes.c_int32),
                ("ksplit", ctypes.c_int32), ("no_pdl", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("test_unarm_first_stage", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


# kamera_reuse_item as a numpy record (32 bytes, naturally aligned)
REUSE_ITEM = np.dtype([("chunk_id", np.int32), ("patch_id", np.int32), ("delta", np.int64), ("seq", np.int32),
                       ("n_tokens", np.int32), ("dst_pos", np.int64)], align=True)
assert REUSE_ITEM.itemsize == 32


class KameraError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{status_string(status)}: {detail}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if build_if_missing:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise ImportError(f"libkamera.so is not built ({_build.LIB}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.c_void_p
        for name in ("kamera_reuse_batched",):
            getattr(lib, name).argtypes = [P, P, P, P, ctypes.c_int32, P, P, P]
        lib.kamera_relocate.argtypes = [P, P, P, ctypes.c_int32, P, P, P]
        lib.kamera_apply_patch.argtypes = [P, P, P, ctypes.c_int32, P, P, P]
        for name in ("kamera_reuse_batched", "kamera_relocate", "kamera_apply_patch"):
            getattr(lib, name).restype = ctypes.c_int
        lib.kamera_factor_workspace_size.argtypes = [P, P]
        lib.kamera_factor_workspace_size.restype = ctypes.c_int
        lib.kamera_factor_patches.argtypes = [P, P, P, ctypes.c_int64, P, ctypes.c_size_t, P]
        lib.kamera_factor_patches.restype = ctypes.c_int
        lib.kamera_factor_patches_noalloc.argtypes = [P, P, P, ctypes.c_int64, P]
        lib.kamera_factor_patches_noalloc.restype = ctypes.c_int
        lib.kamera_orbit_mean.argtypes = [P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, P, P]
        lib.kamera_orbit_mean.restype = ctypes.c_int
        lib.kamera_v_codebook.argtypes = [P, P]
        lib.kamera_v_codebook.restype = ctypes.c_int
        lib.kamera_compress_chunks.argtypes = [P, P, P, P, P]
        lib.kamera_compress_chunks.restype = ctypes.c_int
        lib.kamera_reuse_compressed.argtypes = [P, P, P, P, ctypes.c_int32, P, P, P]
        lib.kamera_reuse_compressed.restype = ctypes.c_int
        lib.kamera_set_launch_tuning.argtypes = [P]
        lib.kamera_set_launch_tuning.restype = ctypes.c_int
        lib.kamera_get_launch_tuning.argtypes = [P]
        lib.kamera_get_launch_tuning.restype = ctypes.c_int
        lib.kamera_status_string.argtypes = [ctypes.c_int]
        lib.kamera_status_string.restype = ctypes.c_char_p
        lib.kamera_last_error.argtypes = []
        lib.kamera_last_error.restype = ctypes.c_char_p
        lib.kamera_abi_version.argtypes = []
        lib.kamera_abi_version.restype = ctypes.c_int32
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().kamera_status_string(int(status)).decode()


def last_error() -> str:
    return load().kamera_last_error().decode()


def abi_version() -> int:
    return int(load().kamera_abi_version())


def _ref(s):
    return None if s is None else ctypes.byref(s)


def kamera_set_launch_tuning(tuning=None, raise_on_error=True, **fields) -> int:
    """Process-wide launch tuning of the reuse entry points (a
    kamera_launch_tuning, or its fields as keywords; neither = defaults)."""
    if tuning is None and fields:
        tuning = kamera_launch_tuning(**fields)
    return _check(load().kamera_set_launch_tuning(_ref(tuning)), raise_on_error)


def kamera_get_launch_tuning() -> kamera_launch_tuning:
    t = kamera_launch_tuning()
    _check(load().kamera_get_launch_tuning(ctypes.byref(t)), True)
    return t


def _check(status: int, raise_on_error: bool) -> int:
    if status != KAMERA_OK and raise_on_error:
        raise KameraError(status, last_error())
    return status


def kamera_reuse_batched(model, store, patches, items_ptr, n_items, pool, err_flag_ptr, stream,
                         raise_on_error=True) -> int:
    st = load().kamera_reuse_batched(_ref(model), _ref(store), _ref(patches), items_ptr, int(n_items), _ref(pool),
                                     err_flag_ptr, stream)
    return _check(st, raise_on_error)


def kamera_relocate(model, store, items_ptr, n_items, pool, err_flag_ptr, stream, raise_on_error=True) -> int:
    st = load().kamera_relocate(_ref(model), _ref(store), items_ptr, int(n_items), _ref(pool), err_flag_ptr, stream)
    return _check(st, raise_on_error)


def kamera_apply_patch(model, patches, items_ptr, n_items, pool, err_flag_ptr, stream, raise_on_error=True) -> int:
    st = load().kamera_apply_patch(_ref(model), _ref(patches), items_ptr, int(n_items), _ref(pool), err_flag_ptr,
                                   stream)
    return _check(st, raise_on_error)


# ---- marshalling helpers (torch tensors -> C structs) -----------------------------------------

def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def model_desc(family, num_layers, num_kv_heads=0, head_dim=0, rope_dim=0, latent_dim=0, pairing=0, patch_frame=0,
               rope_base=10000.0, inv_freq=None, rope_sections=(0, 0, 0), section_delta=None):
    """inv_freq: optional host numpy float64 array kept alive by the returned struct.
    rope_sections: M-RoPE pairs per section; section_delta: device int64
    tensor [n_items][3] of per-section shifts (or None)."""
    m = kamera_model_desc(family, num_layers, num_kv_heads, head_dim, rope_dim, latent_dim, pairing, patch_frame,
                          float(rope_base), None, (ctypes.c_int32 * 3)(*rope_sections), 0, _ptr(section_delta))
    m._keep = section_delta
    if inv_freq is not None:
        arr = np.ascontiguousarray(inv_freq, dtype=np.float64)
        m._inv_freq = arr
        m.inv_freq = arr.ctypes.data
    return m


def chunk_store(data, offset, length):
    """data: bf16 device tensor; offset: int64 device tensor; length: int32 device tensor."""
    s = kamera_chunk_store(_ptr(data), int(data.numel()), _ptr(offset), _ptr(length), int(length.numel()))
    s._keep = (data, offset, length)
    return s


def patch_store(data, offset, length, rank):
    s = kamera_patch_store(_ptr(data), int(data.numel()), _ptr(offset), _ptr(length), int(length.numel()), int(rank))
    s._keep = (data, offset, length)
    return s


def paged_pool(k, v, block_table, page_size):
    """k, v: bf16 [L][num_pages][page_size][D] device tensors (v None for MLA);
    block_table: int32 [n_seqs][max_pages_per_seq] device tensor."""
    p = kamera_paged_pool(_ptr(k), _ptr(v), int(k.shape[1]), int(page_size), _ptr(block_table),
                          int(block_table.shape[0]), int(block_table.shape[1]))
    p._keep = (k, v, block_table)
    return p


def stream_handle(torch_stream=None) -> int:
    import torch

    s = torch_stream if torch_stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def call(mode: str, model, *, items, pool_k, pool_v, block_table, page_size, store=None, store_off=None,
         store_len=None, patch=None, patch_off=None, patch_len=None, rank=0, err_flag=None, stream=None,
         raise_on_error=True) -> int:
    """Marshal device tensors into the C structs and call one entry point.

    mode: "reuse" -> kamera_reuse_batched; "relocate" -> kamera_relocate with
    the chunk store; "relocate_in_place" -> kamera_relocate(store=NULL);
    "apply_patch" -> kamera_apply_patch.  ``items`` is a device uint8/int
    tensor holding kamera_reuse_item records."""
    pool = paged_pool(pool_k, pool_v, block_table, page_size)
    cs = chunk_store(store, store_off, store_len) if store is not None else None
    ps = patch_store(patch, patch_off, patch_len, rank) if (patch is not None and rank) else None
    n_items = int(items.numel() * items.element_size() // REUSE_ITEM.itemsize)
    sh = stream_handle(stream)
    ef = _ptr(err_flag)
    if mode == "reuse":
        return kamera_reuse_batched(model, cs, ps, _ptr(items), n_items, pool, ef, sh, raise_on_error)
    if mode == "relocate":
        return kamera_relocate(model, cs, _ptr(items), n_items, pool, ef, sh, raise_on_error)
    if mode == "relocate_in_place":
        return kamera_relocate(model, None, _ptr(items), n_items, pool, ef, sh, raise_on_error)
    if mode == "apply_patch":
        return kamera_apply_patch(model, ps, _ptr(items), n_items, pool, ef, sh, raise_on_error)
    raise ValueError(f"unknown mode {mode!r}")


# ---- compressed canonical store (PolyKV §2B) -----------------------------------------------------

def kamera_v_codebook():
    """(centroids fp32 [8], thresholds fp32 [7]) of the V codes (a host call)."""
    c = np.zeros(8, np.float32)
    t = np.zeros(7, np.float32)
    _check(load().kamera_v_codebook(c.ctypes.data, t.ctypes.data), True)
    return c, t


def compressed_store(k_codes, k_scale, v_codes, v_norm, row_offset, length):
    """Device tensors: k_codes int8 [rows][D], k_scale fp32 [n_chunks][L], v_codes
    uint8 [rows][H][3*head_dim/8], v_norm fp32 [rows][H], row_offset int64
    [n_chunks], length int32 [n_chunks]."""
    s = kamera_compressed_store(_ptr(k_codes), _ptr(k_scale), _ptr(v_codes), _ptr(v_norm), _ptr(row_offset),
                                _ptr(length), int(length.numel()), 0, int(k_codes.shape[0]))
    s._keep = (k_codes, k_scale, v_codes, v_norm, row_offset, length)
    return s


def kamera_compress_chunks(model, src, dst, err_flag_ptr, stream, raise_on_error=True) -> int:
    return _check(load().kamera_compress_chunks(_ref(model), _ref(src), _ref(dst), err_flag_ptr, stream),
                  raise_on_error)


def kamera_reuse_compressed(model, store, patches, items_ptr, n_items, pool, err_flag_ptr, stream,
                            raise_on_error=True) -> int:
    return _check(load().kamera_reuse_compressed(_ref(model), _ref(store), _ref(patches), items_ptr, n_items,
                                                 _ref(pool), err_flag_ptr, stream), raise_on_error)


def call_compressed(model, cstore, *, items, pool_k, pool_v, block_table, page_size, patch=None, patch_off=None,
                    patch_len=None, rank=0, err_flag=None, stream=None, raise_on_error=True) -> int:
    """kamera_reuse_compressed with device tensors (``cstore`` from compressed_store)."""
    pool = paged_pool(pool_k, pool_v, block_table, page_size)
    ps = patch_store(patch, patch_off, patch_len, rank) if (patch is not None and rank) else None
    n_items = int(items.numel() * items.element_size() // REUSE_ITEM.itemsize)
    return kamera_reuse_compressed(model, cstore, ps, _ptr(items), n_items, pool, _ptr(err_flag),
                                   stream_handle(stream), raise_on_error)


# ---- patch formation ----------------------------------------------------------------------------

def factor_desc(delta, n_slabs, T, D, rank, oversample, power_iters, omega, delta_stride=None):
    """delta: device fp32 [n_slabs][T][D]; omega: device fp32 [D][rank+oversample]."""
    d = kamera_factor_desc(_ptr(delta), int(delta_stride if delta_stride is not None else T * D), int(n_slabs),
                           int(T), int(D), int(rank), int(oversample), int(power_iters), _ptr(omega))
    d._keep = (delta, omega)
    return d


def kamera_factor_workspace_size(desc, raise_on_error=True) -> int:
    out = ctypes.c_size_t(0)
    st = load().kamera_factor_workspace_size(_ref(desc), ctypes.byref(out))
    _check(st, raise_on_error)
    return int(out.value)


def kamera_factor_patches(desc, u_out_ptr, v_out_ptr, out_stride, workspace_ptr, workspace_bytes, stream,
                          raise_on_error=True) -> int:
    st = load().kamera_factor_patches(_ref(desc), u_out_ptr, v_out_ptr, int(out_stride), workspace_ptr,
                                      int(workspace_bytes), stream)
    return _check(st, raise_on_error)


def kamera_factor_patches_noalloc(desc, u_out_ptr, v_out_ptr, out_stride, stream, raise_on_error=True) -> int:
    """Patch formation with the library's static scratch instead of a caller
    workspace, for callers that must not allocate device memory (see the C
    header for the limits and the one-call-at-a-time rule)."""
    st = load().kamera_factor_patches_noalloc(_ref(desc), u_out_ptr, v_out_ptr, int(out_stride), stream)
    return _check(st, raise_on_error)


def kamera_orbit_mean(deltas_ptr, n_orderings, ordering_stride, n_elems, out_ptr, stream, raise_on_error=True) -> int:
    """Mean of deficits sampled under n orderings (the orbit deficit)."""
    st = load().kamera_orbit_mean(deltas_ptr, int(n_orderings), int(ordering_stride), int(n_elems), out_ptr, stream)
    return _check(st, raise_on_error)
