"""fp64 CPU oracle of the Kamera KV-reuse operator (test infrastructure).

TEST INFRASTRUCTURE ONLY: the product path (the CUDA library and its Python
binding) never imports this package.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.

The arithmetic lives in ``kamera_oracle.c`` (plain loops, fp64); this module
compiles it with the host C compiler and marshals numpy arrays through ctypes.
Source of the method: "Kamera: Unified Position-Invariant Multimodal KV Cache
for Training-Free Reuse" (gist.science technical summary), §2 "Methodology:
the Kamera operator" and §3 "window operations".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kamera_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkamera_oracle.so")
_lock = threading.Lock()
_lib = None

MHA, GQA, MLA = 0, 1, 2
ROTATE_HALF, INTERLEAVED = 0, 1
PATCH_AFTER_ROTATION, PATCH_CANONICAL_FRAME = 0, 1
MODE_REUSE, MODE_RELOCATE_IN_PLACE, MODE_PATCH_IN_PLACE = 0, 1, 2
EFLAG_CHUNK_OOB, EFLAG_PAGE_OOB, EFLAG_PATCH_OOB, EFLAG_LEN = 1, 2, 4, 8


class Model(ctypes.Structure):
    _fields_ = [
        ("family", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("rope_dim", ctypes.c_int32),
        ("latent_dim", ctypes.c_int32),
        ("pairing", ctypes.c_int32),
        ("patch_frame", ctypes.c_int32),
        ("sections", ctypes.c_int32 * 3),
    ]


class CStore(ctypes.Structure):
    """A compressed canonical store (see the oracle's "compressed canonical store" section)."""
    _fields_ = [
        ("k_codes", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("v_norm", ctypes.c_void_p),
        ("row_offset", ctypes.c_void_p),
        ("len", ctypes.c_void_p),
        ("n_chunks", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("n_rows", ctypes.c_int64),
        ("codebook", ctypes.c_void_p),
    ]


ITEM_DTYPE = np.dtype(
    [
        ("chunk_id", np.int32),
        ("patch_id", np.int32),
        ("delta", np.int64),
        ("seq", np.int32),
        ("n_tokens", np.int32),
        ("dst_pos", np.int64),
    ],
    align=True,
)
assert ITEM_DTYPE.itemsize == 32


def build_cmd(src: str = _SRC, out: str = _LIB_PATH, cc: str = "gcc") -> list[str]:
    """The compile line: plain -O2, no fast-math, and no contraction of a*b+c
    into a fused multiply-add (the compressed-store encoder's fp32 steps are
    specified operation by operation)."""
    return [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", out, src, "-lm"]


def build(src: str = _SRC, out: str = _LIB_PATH, cc: str = "gcc") -> str:
    """Compile the oracle into a shared library."""
    subprocess.run(build_cmd(src, out, cc), check=True)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  ``path`` selects
    another build of the same source, e.g. a planted-mistake copy in a test."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _declare(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_row_dim.argtypes = [ctypes.POINTER(Model)]
    lib.oracle_row_dim.restype = i32
    lib.oracle_theta.argtypes = [f64, i32, P]
    lib.oracle_theta.restype = None
    lib.oracle_rotate_region.argtypes = [P, i32, P, i64, i32]
    lib.oracle_rotate_region.restype = None
    lib.oracle_rotate_region_sections.argtypes = [P, i32, P, P, P, i32]
    lib.oracle_rotate_region_sections.restype = None
    lib.oracle_rotate_row.argtypes = [ctypes.POINTER(Model), P, i32, P, P]
    lib.oracle_rotate_row.restype = None
    lib.oracle_row.argtypes = [ctypes.POINTER(Model), P, i32, P, i32, P, P, P, i32, P]
    lib.oracle_row.restype = None
    lib.oracle_check_rows.argtypes = [ctypes.POINTER(Model), P, i32, P, i32, i32, P, P, P, i32, P, i32, f64, P, P]
    lib.oracle_check_rows.restype = i64
    lib.oracle_check_rows_compressed.argtypes = [ctypes.POINTER(Model), P, ctypes.POINTER(CStore), i32, i32, i32,
                                                 i32, P, i32, P, P, i32, P, f64, P, P]
    lib.oracle_check_rows_compressed.restype = i64
    lib.oracle_slot.argtypes = [P, i32, i64, i32, i32, i64]
    lib.oracle_slot.restype = i64
    lib.oracle_reuse.argtypes = [ctypes.POINTER(Model), P, i32] + [P, P, P, i32] + [P, P, P, i32, i32] + [
        P, P, i32, P, i32, i32, i64, i32, P, P, P, P, P, P]
    lib.oracle_reuse.restype = i32
    lib.oracle_orbit_mean.argtypes = [P, i32, i64, i64, P]
    lib.oracle_orbit_mean.restype = None
    lib.oracle_jacobi_svd.argtypes = [P, i32, i32, P, P, i32]
    lib.oracle_jacobi_svd.restype = i32
    lib.oracle_lloyd_max_gaussian.argtypes = [i32, i32, P]
    lib.oracle_lloyd_max_gaussian.restype = i32
    lib.oracle_v_codebook.argtypes = [P, P]
    lib.oracle_v_codebook.restype = None
    lib.oracle_quantize_k.argtypes = [P, i64, P, P]
    lib.oracle_quantize_k.restype = None
    lib.oracle_encode_v.argtypes = [P, i32, P, P, P]
    lib.oracle_encode_v.restype = None
    lib.oracle_decode_v.argtypes = [P, ctypes.c_float, i32, P, P]
    lib.oracle_decode_v.restype = None
    lib.oracle_decode_row.argtypes = [ctypes.POINTER(Model), ctypes.POINTER(CStore), i32, i32, i32, i32, P]
    lib.oracle_decode_row.restype = None
    lib.oracle_compress_store.argtypes = [ctypes.POINTER(Model), P, P, P, i32, P, P, P, P, P, P]
    lib.oracle_compress_store.restype = None
    lib.oracle_reuse_compressed.argtypes = [ctypes.POINTER(Model), P, ctypes.POINTER(CStore)] + [
        P, P, P, i32, i32, P, P, i32, P, i32, i32, i64, i32, P, P, P, P, P, P]
    lib.oracle_reuse_compressed.restype = i32
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def model(family, num_layers, num_kv_heads=0, head_dim=0, rope_dim=0, latent_dim=0,
          pairing=ROTATE_HALF, patch_frame=PATCH_AFTER_ROTATION, sections=(0, 0, 0)) -> Model:
    if family != MLA and rope_dim == 0:
        rope_dim = head_dim
    return Model(family, num_layers, num_kv_heads, head_dim, rope_dim, latent_dim, pairing, patch_frame,
                 (ctypes.c_int32 * 3)(*sections))


def _deltas(delta) -> np.ndarray:
    """One shift, or one per M-RoPE section (t, h, w), as int64[3]."""
    d = np.atleast_1d(np.asarray(delta, dtype=np.int64))
    return np.ascontiguousarray(np.resize(d, 3) if d.size == 1 else d[:3])


def row_dim(m: Model) -> int:
    return m.latent_dim + m.rope_dim if m.family == MLA else m.num_kv_heads * m.head_dim


def num_channels(m: Model) -> int:
    return 1 if m.family == MLA else 2


def theta(base: float, rope_dim: int, lib=None) -> np.ndarray:
    lib = lib or load()
    out = np.zeros(rope_dim // 2, np.float64)
    lib.oracle_theta(float(base), int(rope_dim), _ptr(out))
    return out


def rotate_region(x, th, delta: int, pairing=ROTATE_HALF, lib=None) -> np.ndarray:
    """R(delta) on one rotated region (returns a rotated copy, fp64)."""
    lib = lib or load()
    y = np.array(x, dtype=np.float64, copy=True)
    th = _c(th, np.float64)
    lib.oracle_rotate_region(_ptr(y), int(y.shape[0]), _ptr(th), int(delta), int(pairing))
    return y


def rotate_region_sections(x, th, deltas, sections, pairing=ROTATE_HALF, lib=None) -> np.ndarray:
    """R with one shift per M-RoPE section on one rotated region (fp64 copy)."""
    lib = lib or load()
    y = np.array(x, dtype=np.float64, copy=True)
    th = _c(th, np.float64)
    d = _deltas(deltas)
    sec = np.ascontiguousarray(sections, dtype=np.int32)
    lib.oracle_rotate_region_sections(_ptr(y), int(y.shape[0]), _ptr(th), _ptr(d), _ptr(sec), int(pairing))
    return y


def rotate_row(m: Model, th, channel: int, delta, row, lib=None) -> np.ndarray:
    lib = lib or load()
    y = np.array(row, dtype=np.float64, copy=True)
    th = _c(th, np.float64)
    d = _deltas(delta)
    lib.oracle_rotate_row(ctypes.byref(m), _ptr(th), int(channel), _ptr(d), _ptr(y))
    return y


def row(m: Model, th, channel: int, delta, src, u=None, vmat=None, rotate=True, lib=None) -> np.ndarray:
    """One output row: R(delta) src + U V^T row (fp64).  ``u`` [rank], ``vmat`` [D][rank]."""
    lib = lib or load()
    D = row_dim(m)
    src = _c(src, np.float64)
    th = _c(th, np.float64)
    out = np.zeros(D, np.float64)
    rank = 0 if u is None else int(np.asarray(u).shape[0])
    u = _c(u, np.float64)
    vmat = _c(vmat, np.float64) if vmat is not None else np.zeros((D, max(rank, 1)), np.float64)
    d = _deltas(delta)
    lib.oracle_row(ctypes.byref(m), _ptr(th), int(channel), _ptr(d), int(bool(rotate)), _ptr(src), _ptr(u),
                   _ptr(vmat), rank, _ptr(out))
    return out


def check_rows(m: Model, th, channel: int, delta, src_bits, got_bits, u_bits=None, v_bits=None, rotate=True,
               n_exact: int = 0, abs_tol: float = 1e-3, lib=None):
    """Parity of a block of rows against the operator's definition (see
    oracle_check_rows): src_bits, got_bits [n][D] bf16 bits; u_bits [n][rank]
    and v_bits [D][rank] (or None for no patch).  Returns (n_bad, max_err,
    first_bad).  Safe to call from several threads at once (the call releases
    the GIL)."""
    lib = lib or load()
    src = np.ascontiguousarray(src_bits, dtype=np.uint16)
    got = np.ascontiguousarray(got_bits, dtype=np.uint16)
    n, D = src.shape
    assert got.shape == src.shape and D == row_dim(m)
    rank = 0
    if u_bits is not None:
        u_bits = np.ascontiguousarray(u_bits, dtype=np.uint16)
        v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
        rank = int(u_bits.shape[1])
        assert u_bits.shape == (n, rank) and v_bits.shape == (D, rank)
    th = _c(th, np.float64)
    d = _deltas(delta)
    mx = ctypes.c_double(0.0)
    first = ctypes.c_int64(-1)
    bad = lib.oracle_check_rows(ctypes.byref(m), _ptr(th), int(channel), _ptr(d), int(bool(rotate)), int(n),
                                _ptr(src), _ptr(u_bits), _ptr(v_bits), rank, _ptr(got), int(n_exact), float(abs_tol),
                                ctypes.byref(mx), ctypes.byref(first))
    return int(bad), float(mx.value), int(first.value)


def check_rows_compressed(m: Model, th, cs: "Compressed", chunk: int, layer: int, channel: int, t0: int, delta,
                          got_bits, u_bits=None, v_bits=None, abs_tol: float = 1e-3, lib=None):
    """check_rows for rows reused from the compressed store cs: tokens
    t0 .. t0 + n - 1 of (chunk, layer, channel), decoded by the oracle, then
    rotated and patched.  Returns (n_bad, max_err, first_bad)."""
    lib = lib or load()
    got = np.ascontiguousarray(got_bits, dtype=np.uint16)
    n, D = got.shape
    assert D == row_dim(m)
    rank = 0
    if u_bits is not None:
        u_bits = np.ascontiguousarray(u_bits, dtype=np.uint16)
        v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
        rank = int(u_bits.shape[1])
        assert u_bits.shape == (n, rank) and v_bits.shape == (D, rank)
    th = _c(th, np.float64)
    d = _deltas(delta)
    st = cs.struct()
    mx = ctypes.c_double(0.0)
    first = ctypes.c_int64(-1)
    bad = lib.oracle_check_rows_compressed(ctypes.byref(m), _ptr(th), ctypes.byref(st), int(chunk), int(layer),
                                           int(channel), int(t0), _ptr(d), int(n), _ptr(u_bits), _ptr(v_bits), rank,
                                           _ptr(got), float(abs_tol), ctypes.byref(mx), ctypes.byref(first))
    return int(bad), float(mx.value), int(first.value)


def slot(block_table, max_pages_per_seq, num_pages, page_size, seq, pos, lib=None) -> int:
    lib = lib or load()
    bt = _c(block_table, np.int32)
    return int(lib.oracle_slot(_ptr(bt), int(max_pages_per_seq), int(num_pages), int(page_size), int(seq), int(pos)))


def reuse(m: Model, th, mode, *, store=None, store_off=None, store_len=None, patch=None, patch_off=None,
          patch_len=None, rank=0, items, block_table, num_pages, page_size, pool_k_in, pool_v_in=None,
          section_deltas=None, lib=None):
    """The operator over a batch of items into fp64 images of the pool.

    Inputs are bf16 bit patterns as uint16 arrays.  Returns
    ``(err_bits, pool_k_out, pool_v_out, wrote_k, wrote_v)``; the pool images
    have the input pool's shape [L][num_pages][P][D] (fp64) and the masks
    [L][num_pages][P] (uint8)."""
    lib = lib or load()
    th = _c(th, np.float64)
    items = np.ascontiguousarray(items, dtype=ITEM_DTYPE)
    sd = None if section_deltas is None else np.ascontiguousarray(section_deltas, dtype=np.int64).reshape(-1, 3)
    bt = _c(block_table, np.int32)
    n_seqs, max_pages = bt.shape
    pool_k_in = _c(pool_k_in, np.uint16)
    pool_v_in = _c(pool_v_in, np.uint16)
    pk = np.zeros(pool_k_in.shape, np.float64)
    pv = np.zeros(pool_v_in.shape, np.float64) if pool_v_in is not None else None
    rows_shape = pool_k_in.shape[:-1]
    wk = np.zeros(rows_shape, np.uint8)
    wv = np.zeros(rows_shape, np.uint8) if pool_v_in is not None else None
    store = _c(store, np.uint16)
    store_off = _c(store_off, np.int64)
    store_len = _c(store_len, np.int32)
    patch = _c(patch, np.uint16)
    patch_off = _c(patch_off, np.int64)
    patch_len = _c(patch_len, np.int32)
    n_chunks = 0 if store_len is None else int(store_len.shape[0])
    n_patches = 0 if patch_len is None else int(patch_len.shape[0])
    err = lib.oracle_reuse(ctypes.byref(m), _ptr(th), int(mode), _ptr(store), _ptr(store_off), _ptr(store_len),
                           n_chunks, _ptr(patch), _ptr(patch_off), _ptr(patch_len), n_patches, int(rank),
                           _ptr(items), _ptr(sd), int(items.shape[0]), _ptr(bt), int(n_seqs), int(max_pages),
                           int(num_pages), int(page_size), _ptr(pool_k_in), _ptr(pool_v_in), _ptr(pk), _ptr(pv),
                           _ptr(wk), _ptr(wv))
    return int(err), pk, pv, wk, wv


def jacobi_svd(a, max_sweeps: int = 60, lib=None):
    """One-sided Jacobi SVD; returns (U*Sigma [rows][cols], V [cols][cols], sigma)."""
    lib = lib or load()
    a = np.array(a, dtype=np.float64, copy=True, order="C")
    rows, cols = a.shape
    v = np.zeros((cols, cols), np.float64)
    sig = np.zeros(cols, np.float64)
    lib.oracle_jacobi_svd(_ptr(a), rows, cols, _ptr(v), _ptr(sig), int(max_sweeps))
    return a, v, sig


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> fp64 (exact).  Plain widening, kept here so the
    tests' reading of bf16 buffers does not depend on the CUDA path."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def orbit_mean(deltas, lib=None) -> np.ndarray:
    """Mean over the leading axis (the sampled orderings) of fp32 deficits, in fp64."""
    lib = lib or load()
    d = np.ascontiguousarray(deltas, dtype=np.float32)
    n = int(d.shape[0])
    per = int(d.size // max(n, 1))
    out = np.zeros(per, np.float64)
    lib.oracle_orbit_mean(_ptr(d), n, per, per, _ptr(out))
    return out.reshape(d.shape[1:])


# ---- compressed canonical store (PolyKV §2B) ---------------------------------------------------


def lloyd_max_gaussian(levels: int = 8, max_rounds: int = 100000, lib=None):
    """Lloyd-Max centroids of N(0,1) (fp64, ascending) and the rounds used."""
    lib = lib or load()
    c = np.zeros(levels, np.float64)
    rounds = lib.oracle_lloyd_max_gaussian(int(levels), int(max_rounds), _ptr(c))
    return c, int(rounds)


def v_codebook(lib=None):
    """The store format's fp32 codebook (8 centroids) and its 7 thresholds."""
    lib = lib or load()
    c = np.zeros(8, np.float32)
    t = np.zeros(7, np.float32)
    lib.oracle_v_codebook(_ptr(c), _ptr(t))
    return c, t


def quantize_k(x_bits, lib=None):
    """One K tensor (bf16 bits, any shape) -> (int8 codes, fp32 scale)."""
    lib = lib or load()
    x = _c(x_bits, np.uint16)
    q = np.zeros(x.shape, np.int8)
    s = np.zeros(1, np.float32)
    lib.oracle_quantize_k(_ptr(x), int(x.size), _ptr(q), _ptr(s))
    return q, float(s[0])


def encode_v(x_bits, lib=None):
    """Head rows [..., n] (bf16 bits) -> (packed codes [..., 3n/8] uint8, norms [...] fp32)."""
    lib = lib or load()
    x = _c(x_bits, np.uint16)
    n = int(x.shape[-1])
    rows = x.reshape(-1, n)
    _, t32 = v_codebook(lib)
    packed = np.zeros((rows.shape[0], 3 * n // 8), np.uint8)
    norm = np.zeros(rows.shape[0], np.float32)
    for i in range(rows.shape[0]):
        lib.oracle_encode_v(_ptr(rows[i]), n, _ptr(t32), _ptr(packed[i]), _ptr(norm[i:i + 1]))
    return packed.reshape(x.shape[:-1] + (3 * n // 8,)), norm.reshape(x.shape[:-1])


def decode_v(packed, norm, n: int, lib=None) -> np.ndarray:
    """Packed head rows [..., 3n/8] and norms [...] -> decoded rows [..., n] (fp64)."""
    lib = lib or load()
    c32, _ = v_codebook(lib)
    p = _c(packed, np.uint8).reshape(-1, 3 * n // 8)
    nr = np.ascontiguousarray(norm, dtype=np.float32).reshape(-1)
    out = np.zeros((p.shape[0], n), np.float64)
    for i in range(p.shape[0]):
        lib.oracle_decode_v(_ptr(p[i]), float(nr[i]), int(n), _ptr(c32), _ptr(out[i]))
    return out.reshape(np.asarray(packed).shape[:-1] + (n,))


class Compressed:
    """Host arrays of a compressed store (the oracle's layout) plus its ctypes view."""

    def __init__(self, k_codes, k_scale, v_codes, v_norm, row_offset, len_, codebook):
        self.k_codes = np.ascontiguousarray(k_codes, np.int8)
        self.k_scale = np.ascontiguousarray(k_scale, np.float32)
        self.v_codes = np.ascontiguousarray(v_codes, np.uint8)
        self.v_norm = np.ascontiguousarray(v_norm, np.float32)
        self.row_offset = np.ascontiguousarray(row_offset, np.int64)
        self.len = np.ascontiguousarray(len_, np.int32)
        self.codebook = np.ascontiguousarray(codebook, np.float32)

    @property
    def n_rows(self) -> int:
        return int(self.k_codes.shape[0])

    def struct(self) -> CStore:
        return CStore(self.k_codes.ctypes.data, self.k_scale.ctypes.data, self.v_codes.ctypes.data,
                      self.v_norm.ctypes.data, self.row_offset.ctypes.data, self.len.ctypes.data,
                      int(self.len.shape[0]), 0, self.n_rows, self.codebook.ctypes.data)


def compress_store(m: Model, store, store_off, store_len, row_offset=None, n_rows=None, lib=None) -> Compressed:
    """Encode a bf16 chunk store.  Default row layout: the chunks back to back
    (row_offset[c] = sum of L*len over the chunks before c)."""
    lib = lib or load()
    store = _c(store, np.uint16)
    store_off = _c(store_off, np.int64)
    store_len = _c(store_len, np.int32)
    L, D, H, n = m.num_layers, row_dim(m), m.num_kv_heads, m.head_dim
    if row_offset is None:
        row_offset = np.concatenate([[0], np.cumsum(L * store_len.astype(np.int64))[:-1]])
    row_offset = _c(row_offset, np.int64)
    if n_rows is None:
        n_rows = int((row_offset + L * store_len.astype(np.int64)).max(initial=0))
    c32, t32 = v_codebook(lib)
    k_codes = np.zeros((n_rows, D), np.int8)
    k_scale = np.zeros((store_len.shape[0], L), np.float32)
    v_codes = np.zeros((n_rows, H, 3 * n // 8), np.uint8)
    v_norm = np.zeros((n_rows, H), np.float32)
    lib.oracle_compress_store(ctypes.byref(m), _ptr(store), _ptr(store_off), _ptr(store_len),
                              int(store_len.shape[0]), _ptr(row_offset), _ptr(t32), _ptr(k_codes), _ptr(k_scale),
                              _ptr(v_codes), _ptr(v_norm))
    return Compressed(k_codes, k_scale, v_codes, v_norm, row_offset, store_len, c32)


def decode_row(m: Model, cs: Compressed, chunk: int, layer: int, ch: int, t: int, lib=None) -> np.ndarray:
    lib = lib or load()
    out = np.zeros(row_dim(m), np.float64)
    st = cs.struct()
    lib.oracle_decode_row(ctypes.byref(m), ctypes.byref(st), int(chunk), int(layer), int(ch), int(t), _ptr(out))
    return out


def reuse_compressed(m: Model, th, cs: Compressed, *, patch=None, patch_off=None, patch_len=None, rank=0, items,
                     block_table, num_pages, page_size, pool_k_in, pool_v_in, section_deltas=None, lib=None):
    """The reuse operator reading a compressed store; returns like ``reuse``."""
    lib = lib or load()
    th = _c(th, np.float64)
    items = np.ascontiguousarray(items, dtype=ITEM_DTYPE)
    sd = None if section_deltas is None else np.ascontiguousarray(section_deltas, dtype=np.int64).reshape(-1, 3)
    bt = _c(block_table, np.int32)
    n_seqs, max_pages = bt.shape
    pool_k_in = _c(pool_k_in, np.uint16)
    pool_v_in = _c(pool_v_in, np.uint16)
    pk = np.zeros(pool_k_in.shape, np.float64)
    pv = np.zeros(pool_v_in.shape, np.float64)
    wk = np.zeros(pool_k_in.shape[:-1], np.uint8)
    wv = np.zeros(pool_k_in.shape[:-1], np.uint8)
    patch = _c(patch, np.uint16)
    patch_off = _c(patch_off, np.int64)
    patch_len = _c(patch_len, np.int32)
    n_patches = 0 if patch_len is None else int(patch_len.shape[0])
    st = cs.struct()
    err = lib.oracle_reuse_compressed(ctypes.byref(m), _ptr(th), ctypes.byref(st), _ptr(patch), _ptr(patch_off),
                                      _ptr(patch_len), n_patches, int(rank), _ptr(items), _ptr(sd),
                                      int(items.shape[0]), _ptr(bt), int(n_seqs), int(max_pages), int(num_pages),
                                      int(page_size), _ptr(pool_k_in), _ptr(pool_v_in), _ptr(pk), _ptr(pv),
                                      _ptr(wk), _ptr(wv))
    return int(err), pk, pv, wk, wv
