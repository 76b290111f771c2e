"""Pins of the oracle's compressed canonical store (CPU only).

Source: "PolyKV" (gist.science summary, Spanish edition), §2B: K as int8
with one linear scale per tensor; V at 3 bits by TurboQuant MSE -- a fast
Walsh-Hadamard rotation, the Lloyd-Max centroids of N(0,1), and decoding by
centroid values plus the inverse transform; ratio 16 / ((8 + 3) / 2) = 2.91.

Each oracle function is checked against something other than itself: Max's
1960 table and numerical integration for the codebook, the error bound and
scale invariance for the int8 codes, scipy's Hadamard matrix and a closed
form for the V codec, the Lloyd-Max distortion for Gaussian rows, and an
independent vectorised formulation for the reuse operator over a compressed
store.
"""
import json
import os

import numpy as np
import pytest
from scipy import integrate, linalg, stats

import oracle
from synth import gen
from synth import workloads as W
from tests.test_oracle_operator import _bits_to_f64, _complex_rotate_rows, _theta_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    return json.load(open(os.path.join(GOLDEN, name)))


# ---- the codebook -------------------------------------------------------------------------------

def test_lloyd_max_matches_max_1960_table(oracle_lib):
    g = _golden("lloyd_max_gaussian_n8.json")
    c, rounds = oracle.lloyd_max_gaussian(8)
    assert rounds < 100000
    np.testing.assert_allclose(c[4:], g["positive_outputs"], atol=g["abs_tol"])
    np.testing.assert_allclose(-c[:4][::-1], g["positive_outputs"], atol=g["abs_tol"])
    t = 0.5 * (c[1:] + c[:-1])
    np.testing.assert_allclose(t[3:], g["positive_thresholds"], atol=g["abs_tol"])


def test_lloyd_max_optimality_by_quadrature(oracle_lib):
    """Each centroid is the mean of N(0,1) over its cell (integrated
    numerically), and the distortion is Max's value."""
    g = _golden("lloyd_max_gaussian_n8.json")
    c, _ = oracle.lloyd_max_gaussian(8)
    edges = np.concatenate([[-np.inf], 0.5 * (c[1:] + c[:-1]), [np.inf]])
    pdf = stats.norm.pdf
    mse = 0.0
    for k in range(8):
        a, b = edges[k], edges[k + 1]
        mass = integrate.quad(pdf, a, b, epsabs=1e-14, epsrel=1e-13)[0]
        first = integrate.quad(lambda z: z * pdf(z), a, b, epsabs=1e-14, epsrel=1e-13)[0]
        assert abs(first / mass - c[k]) < 1e-9
        mse += integrate.quad(lambda z: (z - c[k]) ** 2 * pdf(z), a, b, epsabs=1e-14, epsrel=1e-13)[0]
    assert abs(mse - g["mean_squared_error"]) < g["mse_abs_tol"]


def test_codebook_is_fp32_antisymmetric_with_midpoint_thresholds(oracle_lib):
    c64, _ = oracle.lloyd_max_gaussian(8)
    c32, t32 = oracle.v_codebook()
    assert c32.dtype == np.float32 and t32.dtype == np.float32
    np.testing.assert_array_equal(c32[4:], c64[4:].astype(np.float32))
    np.testing.assert_array_equal(c32[:4], -c32[4:][::-1])
    assert np.all(np.diff(c32) > 0)
    np.testing.assert_array_equal(t32, ((c32[1:] + c32[:-1]) * np.float32(0.5)).astype(np.float32))
    assert t32[3] == 0.0


# ---- K: int8, one scale per tensor -------------------------------------------------------------------

def _bf16(x):
    return gen.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_k_codes_within_half_a_step_and_full_range(oracle_lib):
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((64, 96)) * 3.0)
    xf = _bits_to_f64(x)
    q, s = oracle.quantize_k(x)
    assert q.dtype == np.int8 and np.abs(q).max() == 127
    i = np.unravel_index(np.abs(xf).argmax(), xf.shape)
    assert abs(int(q[i])) == 127 and np.sign(q[i]) == np.sign(xf[i])
    assert abs(s - np.abs(xf).max() / 127) <= 1e-6 * s
    assert np.all(np.abs(xf - q.astype(np.float64) * s) <= 0.5 * s * (1 + 1e-5))
    assert np.all(np.abs(q) <= 127)


def test_k_codes_invariant_under_power_of_two_scaling(oracle_lib):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(500).astype(np.float32)
    q1, s1 = oracle.quantize_k(_bf16(x))
    q2, s2 = oracle.quantize_k(_bf16(x * 8.0))
    np.testing.assert_array_equal(q1, q2)
    assert s2 == 8.0 * s1


def test_k_zero_tensor_gives_zero_codes_and_scale(oracle_lib):
    q, s = oracle.quantize_k(np.zeros(100, np.uint16))
    assert s == 0.0 and not q.any()


# ---- V: Walsh-Hadamard rotation + 3-bit Lloyd-Max codes ----------------------------------------

def _unpack(packed, n):
    """Codes from the format's definition: 6-bit field i = code[i] | code[i + n/2] << 3 at bit 6i."""
    bits = np.unpackbits(np.asarray(packed, np.uint8), bitorder="little")
    codes = np.zeros(n, np.int64)
    for i in range(n // 2):
        f = sum(int(bits[6 * i + b]) << b for b in range(6))
        codes[i], codes[i + n // 2] = f & 7, f >> 3
    return codes


def _pack(codes):
    n = len(codes)
    bits = np.zeros(3 * n, np.uint8)
    for i in range(n // 2):
        f = int(codes[i]) | int(codes[i + n // 2]) << 3
        for b in range(6):
            bits[6 * i + b] = (f >> b) & 1
    return np.packbits(bits, bitorder="little")


@pytest.mark.parametrize("n", [64, 128])
def test_decode_is_scaled_hadamard_of_centroids(oracle_lib, n):
    rng = np.random.default_rng(n)
    c32, _ = oracle.v_codebook()
    Hm = linalg.hadamard(n).astype(np.float64)
    for _ in range(5):
        codes = rng.integers(0, 8, n)
        norm = np.float32(rng.uniform(0.5, 4.0))
        got = oracle.decode_v(_pack(codes)[None], np.array([norm]), n)[0]
        want = float(norm) / n * (Hm @ c32[codes].astype(np.float64))
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n", [64, 128])
def test_encode_picks_the_nearest_centroid_of_the_normalised_coordinate(oracle_lib, n):
    """z = (H x) / ||x|| computed in fp64 with scipy's Hadamard matrix; the
    code is the nearest centroid, except where z lies within fp32 rounding of
    a threshold (there either neighbour is accepted)."""
    rng = np.random.default_rng(10 + n)
    c32, t32 = oracle.v_codebook()
    Hm = linalg.hadamard(n).astype(np.float64)
    x = _bf16(rng.standard_normal((40, n)) * rng.uniform(0.1, 10.0, (40, 1)))
    packed, norms = oracle.encode_v(x)
    xf = _bits_to_f64(x)
    for r in range(40):
        codes = _unpack(packed[r], n)
        assert abs(norms[r] - np.linalg.norm(xf[r])) <= 1e-6 * np.linalg.norm(xf[r])
        z = Hm @ xf[r] / np.linalg.norm(xf[r])
        near = np.abs(z[:, None] - c32[None, :].astype(np.float64)).argmin(axis=1)
        tie = np.min(np.abs(z[:, None] - t32[None, :].astype(np.float64)), axis=1) < 1e-5
        assert np.all((codes == near) | (tie & (np.abs(codes - near) == 1)))


def test_one_hot_row_decodes_to_the_centroid_at_one(oracle_lib):
    """x = e_0: H x is all ones and ||x|| = 1, so every z is 1 -> code 5 (the
    centroid 0.756, since 0.5006 <= 1 < 1.050); decoding gives c_5 * e_0."""
    n = 128
    c32, _ = oracle.v_codebook()
    x = np.zeros(n, np.float32)
    x[0] = 1.0
    packed, norms = oracle.encode_v(_bf16(x)[None])
    assert (_unpack(packed[0], n) == 5).all() and norms[0] == 1.0
    y = oracle.decode_v(packed, norms, n)[0]
    want = np.zeros(n)
    want[0] = c32[5]
    np.testing.assert_allclose(y, want, atol=1e-12)


def test_zero_row_encodes_to_zero(oracle_lib):
    packed, norms = oracle.encode_v(np.zeros((1, 128), np.uint16))
    assert norms[0] == 0.0 and not packed.any()
    assert not oracle.decode_v(packed, norms, 128).any()


def test_gaussian_rows_lose_the_lloyd_max_distortion(oracle_lib):
    """For iid Gaussian rows the normalised coordinates are close to N(0,1),
    so ||x - x^||^2 / ||x||^2 averages Max's distortion 0.0345."""
    g = _golden("lloyd_max_gaussian_n8.json")
    n = 128
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((600, n)))
    packed, norms = oracle.encode_v(x)
    y = oracle.decode_v(packed, norms, n)
    xf = _bits_to_f64(x)
    rel = np.sum((xf - y) ** 2, axis=1) / np.sum(xf ** 2, axis=1)
    assert abs(rel.mean() - g["mean_squared_error"]) < 0.002


def test_byte_budget_gives_the_pages_ratio(oracle_lib):
    g = _golden("polykv_ratio.json")
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=40, rank=0, page_size=16)
    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim)
    cs = oracle.compress_store(m, wl.host_store(), wl.store_off, np.array(wl.chunk_lens, np.int32))
    bf16_bytes = wl.store_elems * 2
    ratio = bf16_bytes / (cs.k_codes.nbytes + cs.v_codes.nbytes)
    assert abs(ratio - g["ratio"]) < g["abs_tol"]
    assert abs(g["baseline_bits"] / ((g["k_bits"] + g["v_bits"]) / 2) - g["ratio"]) < g["abs_tol"]


def check_store_encoding(wl, cs):
    """Every (chunk, layer) K tensor and every V head row of the bf16 store
    against its place in the compressed store, by properties of the codecs
    computed here with numpy and scipy: the K scale is max|x| / 127, every K
    code lies within half a step of its value and the largest |x| takes
    +-127; each V norm is the row's Euclidean norm, each V code the nearest
    centroid of (H x) / ||x|| (either neighbour within fp32 rounding of a
    threshold)."""
    T_all, D, H, n, L = wl.chunk_lens, wl.D, wl.num_kv_heads, wl.head_dim, wl.num_layers
    store = wl.host_store()
    Hm = linalg.hadamard(n).astype(np.float64)
    c64 = cs.codebook.astype(np.float64)
    for c, T in enumerate(T_all):
        for l in range(L):
            base = int(wl.store_off[c]) + 2 * l * T * D
            k = _bits_to_f64(store[base:base + T * D]).reshape(T, D)
            v = _bits_to_f64(store[base + T * D:base + 2 * T * D]).reshape(T, D)
            r0 = int(cs.row_offset[c]) + l * T
            s = float(cs.k_scale[c, l])
            assert abs(s - np.abs(k).max() / 127) <= 1e-6 * s
            q = cs.k_codes[r0:r0 + T].astype(np.float64)
            assert np.all(np.abs(k - q * s) <= 0.5 * s * (1 + 1e-5))
            i = np.unravel_index(np.abs(k).argmax(), k.shape)
            assert abs(q[i]) == 127
            for t in range(T):
                for h in range(H):
                    x = v[t, h * n:(h + 1) * n]
                    nx = np.linalg.norm(x)
                    assert abs(float(cs.v_norm[r0 + t, h]) - nx) <= 1e-6 * nx
                    z = Hm @ x / nx
                    near = np.abs(z[:, None] - c64[None, :]).argmin(axis=1)
                    dist = np.abs(z[:, None] - (c64[1:] + c64[:-1])[None, :] / 2).min(axis=1)
                    codes = _unpack(cs.v_codes[r0 + t, h], n)
                    assert np.all((codes == near) | ((dist < 1e-5) & (np.abs(codes - near) == 1)))


def test_compressed_store_holds_each_tensor_and_head_row_in_place(oracle_lib):
    """The store layout (row_offset[c] + l*T + t; K scale per (chunk, layer);
    V head rows in order) and the codecs, for two chunks of three layers
    whose rows start after a gap and leave another gap between them."""
    wl = W.gqa_video(num_layers=3, n_chunks=2, T=24, rank=0, page_size=16)
    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim)
    lens = np.array(wl.chunk_lens, np.int32)
    row_offset = np.array([5, 5 + wl.num_layers * int(lens[0]) + 7], np.int64)
    cs = oracle.compress_store(m, wl.host_store(), wl.store_off, lens, row_offset=row_offset)
    check_store_encoding(wl, cs)
    assert not cs.k_codes[:5].any() and not cs.v_norm[:5].any()


# ---- the reuse operator reading a compressed store -----------------------------------------------------

def _decode_np(wl, cs, chunk, layer, ch):
    """Rows [T][D] of (chunk, layer, channel) decoded with numpy and scipy's Hadamard matrix."""
    T, D, H, n = wl.chunk_lens[chunk], wl.D, wl.num_kv_heads, wl.head_dim
    r0 = int(cs.row_offset[chunk]) + layer * T
    if ch == 0:
        return cs.k_codes[r0:r0 + T].astype(np.float64) * float(cs.k_scale[chunk, layer])
    Hm = linalg.hadamard(n).astype(np.float64)
    out = np.zeros((T, D))
    for t in range(T):
        for h in range(H):
            codes = _unpack(cs.v_codes[r0 + t, h], n)
            out[t, h * n:(h + 1) * n] = float(cs.v_norm[r0 + t, h]) / n * (Hm @ cs.codebook[codes].astype(np.float64))
    return out


def _independent_reuse_compressed(wl, cs):
    theta = _theta_np(wl.rope_base, wl.rope_dim)
    pk = _bits_to_f64(wl.host_pool(0))
    pv = _bits_to_f64(wl.host_pool(1))
    wk = np.zeros(pk.shape[:-1], bool)
    wv = np.zeros(pk.shape[:-1], bool)
    for i_it, it in enumerate(wl.items):
        T, c, p, delta = int(it["n_tokens"]), int(it["chunk_id"]), int(it["patch_id"]), int(it["delta"])
        if sum(wl.rope_sections) and wl.section_deltas is not None:
            delta = np.repeat(np.asarray(wl.section_deltas[i_it], np.float64), wl.rope_sections)
        pos = int(it["dst_pos"]) + np.arange(T)
        pages, slots = wl.block_table[int(it["seq"]), pos // wl.page_size], pos % wl.page_size
        for layer in range(wl.num_layers):
            for ch in range(2):
                x = _decode_np(wl, cs, c, layer, ch)
                patch = 0.0
                if wl.rank and p >= 0:
                    patch = _bits_to_f64(wl.u_rows(p, layer, ch)) @ _bits_to_f64(wl.v_rows(p, layer, ch)).T
                if ch == 0 and wl.patch_frame == W.CANONICAL_FRAME:
                    y = _complex_rotate_rows(x + patch, wl.num_kv_heads, wl.rope_dim, wl.head_dim, 0, delta, theta,
                                             wl.pairing)
                elif ch == 0:
                    y = _complex_rotate_rows(x, wl.num_kv_heads, wl.rope_dim, wl.head_dim, 0, delta, theta,
                                             wl.pairing) + patch
                else:
                    y = x + patch
                (pk if ch == 0 else pv)[layer, pages, slots] = y
                (wk if ch == 0 else wv)[layer, pages, slots] = True
    return pk, pv, wk, wv


def _cases():
    small = W.gqa_video(num_layers=2, n_chunks=3, T=37, rank=16, page_size=16)
    return {"encoded": (small, "encode"), "random_contents": (small, "random"),
            "mha64_rank0": (W.tiny_mha().replace(rank=0, patch_lens=[], items=W.tiny_mha().items.copy()),
                            "encode")}


def _store_for(wl, how):
    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim)
    if how == "encode":
        return m, oracle.compress_store(m, wl.host_store(), wl.store_off, np.array(wl.chunk_lens, np.int32))
    r = wl.random_compressed()
    c32, _ = oracle.v_codebook()
    return m, oracle.Compressed(r["k_codes"], r["k_scale"], r["v_codes"], r["v_norm"], r["row_offset"], r["len"],
                                c32)


@pytest.mark.parametrize("case", ["encoded", "random_contents", "mha64_rank0"])
def test_reuse_compressed_matches_independent_formulation(oracle_lib, case):
    wl, how = _cases()[case]
    if wl.rank == 0:
        wl.items["patch_id"] = -1
    m, cs = _store_for(wl, how)
    th = oracle.theta(wl.rope_base, wl.rope_dim)
    kw = {}
    if wl.rank:
        kw = dict(patch=wl.host_patch(), patch_off=wl.patch_off, patch_len=np.array(wl.patch_lens, np.int32),
                  rank=wl.rank)
    err, pk, pv, wk, wv = oracle.reuse_compressed(m, th, cs, items=wl.items, block_table=wl.block_table,
                                                  num_pages=wl.num_pages, page_size=wl.page_size,
                                                  pool_k_in=wl.host_pool(0), pool_v_in=wl.host_pool(1), **kw)
    assert err == 0
    ik, iv, iwk, iwv = _independent_reuse_compressed(wl, cs)
    np.testing.assert_array_equal(wk.astype(bool), iwk)
    np.testing.assert_array_equal(wv.astype(bool), iwv)
    np.testing.assert_allclose(pk[iwk], ik[iwk], rtol=0, atol=1e-10)
    np.testing.assert_allclose(pv[iwv], iv[iwv], rtol=0, atol=1e-10)
    assert np.isnan(pk[~iwk]).all() and np.isnan(pv[~iwv]).all()


def test_reuse_compressed_error_bits(oracle_lib):
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=24, rank=0, page_size=16)
    wl.items["patch_id"] = -1
    m, cs = _store_for(wl, "random")
    th = oracle.theta(wl.rope_base, wl.rope_dim)

    def run(items, cs=cs):
        return oracle.reuse_compressed(m, th, cs, items=items, block_table=wl.block_table, num_pages=wl.num_pages,
                                       page_size=wl.page_size, pool_k_in=wl.host_pool(0),
                                       pool_v_in=wl.host_pool(1))[0]

    bad = wl.items.copy()
    bad["chunk_id"][0] = 7
    assert run(bad) == oracle.EFLAG_CHUNK_OOB
    bad = wl.items.copy()
    bad["n_tokens"][0] = 23
    assert run(bad) == oracle.EFLAG_LEN
    short = oracle.Compressed(cs.k_codes[:-1], cs.k_scale, cs.v_codes[:-1], cs.v_norm[:-1], cs.row_offset, cs.len,
                              cs.codebook)
    assert run(wl.items, short) == oracle.EFLAG_CHUNK_OOB  # the last chunk's rows run past the store


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_compressed_workloads_match_independent_formulation(oracle_lib, seed):
    """The seeded random batches of the GPU fuzz of the compressed store (the
    oracle's encoding for even seeds, random contents for odd ones) through
    the oracle and through the independent formulation."""
    from tests import harness as H
    from tests.test_gpu_fuzz import random_workload

    wl = random_workload(3000 + seed, compressed=True)
    if seed % 2 == 0:
        m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim)
        cs = oracle.compress_store(m, wl.host_store(), wl.store_off, np.array(wl.chunk_lens, np.int32),
                                   row_offset=wl.comp_row_offset, n_rows=wl.comp_rows)
    else:
        cs = H.oracle_store(H.comp_arrays(wl.random_compressed()))
    err, pk, pv, wk, wv = H.oracle_reference_compressed(wl, cs)
    assert err == 0
    ik, iv, iwk, iwv = _independent_reuse_compressed(wl, cs)
    for got, want, w, iw in ((pk, ik, wk, iwk), (pv, iv, wv, iwv)):
        np.testing.assert_array_equal(w.astype(bool), iw)
        np.testing.assert_allclose(got[iw], want[iw], rtol=0, atol=1e-9)
        np.testing.assert_array_equal(got[~iw], want[~iw])
