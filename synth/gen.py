"""Seeded, counter-based synthetic inputs (host side, numpy).

This module holds no arithmetic of the reuse operator: it only draws the
numbers that go INTO it (canonical K/V rows, patch factors, pool contents,
deltas, block tables).  Both the CUDA path and the oracle consume what it
makes.  A device twin (``synth_cuda.cu``) produces the same bits on the GPU
for the multi-GB stores; a GPU test checks the two bit for bit.

Generator.  Every value is a pure function of (stream, index):

    splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): the n-th output of a generator seeded with s is
    mix(s + (n + 1) * 0x9E3779B97F4A7C15) with the published finaliser
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
        z = (z ^ (z >> 27)) * 0x94D049BB133111EB
        z =  z ^ (z >> 31)

Normal variates use the Irwin-Hall sum of the four 16-bit fields of one
output: s in [0, 262140], mean 131070, variance (2^32 - 1) / 3.  The value
is fp32(s - 131070) * fp32(sigma / sd) (one fp32 multiply, round to nearest
even), rounded to bf16 (round to nearest even).  Tails stop at about 3.46 sd.
"""
from __future__ import annotations

import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
IH_MEAN = 131070
IH_SD = math.sqrt((2.0**32 - 1.0) / 3.0)

# index layout shared by host and device generators
T_BITS = 20  # token index stride: 2^20 tokens per (chunk, layer, channel)
D_BITS = 11  # feature index stride: 2^11 features per row
R_BITS = 6  # rank index stride: 64

STREAM_KV, STREAM_U, STREAM_V, STREAM_POOL, STREAM_OUTLIER, STREAM_DELTA, STREAM_PERM = 1, 2, 3, 4, 5, 6, 7


def mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
    return z ^ (z >> np.uint64(31))


def hash64(stream: int, idx) -> np.ndarray:
    """The idx-th output (0-based) of splitmix64 seeded with ``stream``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(stream) + (idx + np.uint64(1)) * GOLDEN
    return mix64(z)


def stream_id(seed: int, tag: int) -> int:
    """Seed of one named stream: splitmix64 output of (seed, tag)."""
    return int(hash64(seed & 0xFFFFFFFFFFFFFFFF, np.uint64(tag)))


def scale_f32(sigma: float) -> np.float32:
    """The fp32 multiplier that maps an Irwin-Hall integer to N(0, sigma)."""
    return np.float32(sigma / IH_SD)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (inputs are finite)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = u + np.uint32(0x7FFF) + lsb
    return (r >> np.uint32(16)).astype(np.uint16)


def normal_bits(stream: int, idx, scale: np.float32) -> np.ndarray:
    """bf16 bits of N(0, sigma) variates at counter positions ``idx``."""
    h = hash64(stream, idx)
    m = np.uint64(0xFFFF)
    s = (h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m) + (h >> np.uint64(48))
    x = (s.astype(np.int64) - IH_MEAN).astype(np.float32)
    return f32_to_bf16_bits(x * np.float32(scale))


def fill_rows(stream: int, rows: int, row_len: int, idx0: int, idx_row_stride: int, scale: np.float32,
              outlier_stream: int = 0, okey0: int = 0, outlier_scale: np.float32 | None = None,
              outlier_permille: int = 0) -> np.ndarray:
    """[rows][row_len] bf16 bits; element (r, j) draws counter idx0 + r*stride + j.

    If ``outlier_permille`` > 0, feature j is an outlier channel (drawn with
    ``outlier_scale``) when hash64(outlier_stream, okey0 + j) % 1000 is below
    it -- the same channels for every row of the block."""
    r = np.arange(rows, dtype=np.uint64)[:, None]
    j = np.arange(row_len, dtype=np.uint64)[None, :]
    with np.errstate(over="ignore"):
        idx = np.uint64(idx0) + r * np.uint64(idx_row_stride) + j
    h = hash64(stream, idx)
    m = np.uint64(0xFFFF)
    s = (h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m) + (h >> np.uint64(48))
    x = (s.astype(np.int64) - IH_MEAN).astype(np.float32)
    sc = np.full((1, row_len), np.float32(scale), np.float32)
    if outlier_permille > 0:
        hk = hash64(outlier_stream, np.uint64(okey0) + np.arange(row_len, dtype=np.uint64))
        sel = (hk % np.uint64(1000)) < np.uint64(outlier_permille)
        sc[0, sel] = np.float32(outlier_scale)
    return f32_to_bf16_bits(x * sc)


# ---- index helpers (the counter layout of each tensor kind) -----------------

def kv_index(chunk: int, layer: int, channel: int, token: int = 0, feature: int = 0) -> int:
    slab = (chunk * 128 + layer) * 2 + channel
    return (((slab << T_BITS) + token) << D_BITS) + feature


def u_index(patch: int, layer: int, channel: int, token: int = 0, r: int = 0) -> int:
    slab = (patch * 128 + layer) * 2 + channel
    return (((slab << T_BITS) + token) << R_BITS) + r


def v_index(patch: int, layer: int, channel: int, feature: int = 0, r: int = 0) -> int:
    slab = (patch * 128 + layer) * 2 + channel
    return (((slab << D_BITS) + feature) << R_BITS) + r


def pool_index(layer: int, page: int, slot: int = 0, feature: int = 0) -> int:
    return (((((layer << 24) + page) << 8) + slot) << D_BITS) + feature


def outlier_key(layer: int, channel: int) -> int:
    return (layer * 2 + channel) << D_BITS


def uniform_int(stream: int, idx, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi] (modulo bias < 2^-40 for the ranges used)."""
    h = hash64(stream, idx)
    return (h % np.uint64(hi - lo + 1)).astype(np.int64) + lo


def permutation(stream: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n): argsort of the hashes (stable)."""
    return np.argsort(hash64(stream, np.arange(n, dtype=np.uint64)), kind="stable").astype(np.int64)


def normal_f32(stream: int, idx, sigma: float = 1.0) -> np.ndarray:
    """fp32 N(0, sigma) variates at counter positions idx (the Irwin-Hall value
    before any bf16 rounding)."""
    h = hash64(stream, idx)
    m = np.uint64(0xFFFF)
    s = (h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m) + (h >> np.uint64(48))
    return (s.astype(np.int64) - IH_MEAN).astype(np.float32) * scale_f32(sigma)


STREAM_OMEGA, STREAM_DEFICIT = 8, 9


def gaussian_test_matrix(seed: int, D: int, k: int) -> np.ndarray:
    """Omega [D][k] fp32 N(0,1): the randomized range finder's test matrix."""
    return normal_f32(stream_id(seed, STREAM_OMEGA), np.arange(D * k, dtype=np.uint64)).reshape(D, k)


def low_rank_deficit(seed: int, slab: int, T: int, D: int, spectrum, noise: float = 0.0) -> np.ndarray:
    """A synthetic deficit [T][D] fp32: A diag(spectrum) B^T / sqrt(T D) + noise
    with A, B Gaussian -- a low-rank matrix with the given (approximate)
    singular values plus a small full-rank floor."""
    r = len(spectrum)
    st = stream_id(seed, STREAM_DEFICIT)
    base = np.uint64(slab) << np.uint64(40)
    A = normal_f32(st, base + np.arange(T * r, dtype=np.uint64)).reshape(T, r).astype(np.float64)
    B = normal_f32(st, base + np.uint64(1 << 36) + np.arange(D * r, dtype=np.uint64)).reshape(D, r).astype(np.float64)
    out = (A * np.asarray(spectrum, np.float64)) @ B.T / np.sqrt(T * D)
    if noise:
        N = normal_f32(st, base + np.uint64(1 << 38) + np.arange(T * D, dtype=np.uint64)).reshape(T, D)
        out = out + noise * N / np.sqrt(max(T, D))
    return out.astype(np.float32)


# ---- random compressed-store contents (bytes and positive scales; no encoding) ----------------

STREAM_KCODE, STREAM_VCODE, STREAM_KSCALE, STREAM_VNORM = 10, 11, 12, 13


def random_bytes(stream: int, n: int, idx0: int = 0) -> np.ndarray:
    """n uniform bytes: the little-endian bytes of hash64 at idx0, idx0 + 1, ..."""
    words = hash64(stream, np.uint64(idx0) + np.arange((n + 7) // 8, dtype=np.uint64))
    return words.astype("<u8").view(np.uint8)[:n].copy()


def uniform_f32(stream: int, idx, lo: float, hi: float) -> np.ndarray:
    """fp32 uniform in [lo, hi) from the top 24 bits of hash64."""
    h = hash64(stream, idx) >> np.uint64(40)
    return (lo + (hi - lo) * (h.astype(np.float64) / float(1 << 24))).astype(np.float32)
