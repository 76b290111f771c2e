"""Pins of the oracle's whole-batch operator (gather -> R(delta) -> + U V^T ->
paged scatter) against an independent vectorised formulation, the pool's
untouched slots, and the error-bit convention (CPU only).

Kamera §2 reuse equation; §3 window operations (reorder, sliding-window
survival with R(delta) only, recall with a fresh patch).
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W


def _theta_np(base, d):
    return np.exp(-np.log(base) * np.arange(0, d, 2) / d)


def _bits_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _oracle_model(wl):
    return oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim, wl.latent_dim,
                        wl.pairing, wl.patch_frame)


def _run_oracle(wl, pool_k=None, pool_v=None, lib=None):
    m = _oracle_model(wl)
    th = oracle.theta(wl.rope_base, wl.rope_dim, lib=lib)
    mode = {"reuse": oracle.MODE_REUSE, "relocate_in_place": oracle.MODE_RELOCATE_IN_PLACE,
            "apply_patch": oracle.MODE_PATCH_IN_PLACE}[wl.mode]
    pool_k = wl.host_pool(0) if pool_k is None else pool_k
    pool_v = (wl.host_pool(1) if pool_v is None else pool_v) if wl.n_ch == 2 else None
    kw = {}
    if wl.mode == "reuse":
        kw.update(store=wl.host_store(), store_off=wl.store_off, store_len=np.array(wl.chunk_lens, np.int32))
    if wl.rank:
        kw.update(patch=wl.host_patch(), patch_off=wl.patch_off, patch_len=np.array(wl.patch_lens, np.int32),
                  rank=wl.rank)
    return oracle.reuse(m, th, mode, items=wl.items, block_table=wl.block_table, num_pages=wl.num_pages,
                        page_size=wl.page_size, pool_k_in=pool_k, pool_v_in=pool_v, lib=lib, **kw)


def _complex_rotate_rows(x, heads, rope, stride, col0, delta, theta, pairing):
    """Rotate [T][D] rows by delta with complex arithmetic, vectorised."""
    y = x.copy()
    e = np.exp(1j * delta * theta)
    for h in range(heads):
        a = col0 + h * stride
        seg = x[:, a:a + rope]
        if pairing == W.ROTATE_HALF:
            z = (seg[:, :rope // 2] + 1j * seg[:, rope // 2:]) * e
            y[:, a:a + rope // 2], y[:, a + rope // 2:a + rope] = z.real, z.imag
        else:
            z = (seg[:, 0::2] + 1j * seg[:, 1::2]) * e
            y[:, a:a + rope:2], y[:, a + 1:a + rope:2] = z.real, z.imag
    return y


def _independent_reuse(wl):
    """The same operator as matrix algebra over whole slabs + explicit page map
    (M-RoPE: a per-pair shift vector from the sections)."""
    D, L = wl.D, wl.num_layers
    theta = _theta_np(wl.rope_base, wl.rope_dim)
    pk = _bits_to_f64(wl.host_pool(0))
    pv = _bits_to_f64(wl.host_pool(1)) if wl.n_ch == 2 else None
    wk = np.zeros(pk.shape[:-1], bool)
    wv = np.zeros(pk.shape[:-1], bool)
    for i_it, it in enumerate(wl.items):
        T, c, p, delta = int(it["n_tokens"]), int(it["chunk_id"]), int(it["patch_id"]), int(it["delta"])
        if sum(wl.rope_sections) and wl.section_deltas is not None:
            # M-RoPE: pair i turns by the shift of the section it falls in
            delta = np.repeat(np.asarray(wl.section_deltas[i_it], np.float64), wl.rope_sections)
        pos = int(it["dst_pos"]) + np.arange(T)
        pages = wl.block_table[int(it["seq"]), pos // wl.page_size]
        slots = pos % wl.page_size
        for layer in range(L):
            for ch in range(wl.n_ch):
                x = _bits_to_f64(wl.store_rows(c, layer, ch))
                if wl.rank and p >= 0:
                    U = _bits_to_f64(wl.u_rows(p, layer, ch))
                    V = _bits_to_f64(wl.v_rows(p, layer, ch))
                    patch = U @ V.T
                else:
                    patch = 0.0
                if ch == 0:
                    if wl.family == W.MLA:
                        heads, stride, col0 = 1, 0, wl.latent_dim
                    else:
                        heads, stride, col0 = wl.num_kv_heads, wl.head_dim, 0
                    if wl.patch_frame == W.CANONICAL_FRAME:
                        y = _complex_rotate_rows(x + patch, heads, wl.rope_dim, stride, col0, delta, theta,
                                                 wl.pairing)
                    else:
                        y = _complex_rotate_rows(x, heads, wl.rope_dim, stride, col0, delta, theta,
                                                 wl.pairing) + patch
                else:
                    y = x + patch
                dst = pk if ch == 0 else pv
                dst[layer, pages, slots] = y
                (wk if ch == 0 else wv)[layer, pages, slots] = True
    return pk, pv, wk, wv


def _small_gqa(**kw):
    wl = W.gqa_video(num_layers=2, n_chunks=3, T=70, rank=16, page_size=16)
    return wl.replace(**kw) if kw else wl


CASES = {
    "gqa_rank16": lambda: _small_gqa(),
    "gqa_interleaved_canonical": lambda: _small_gqa(pairing=W.INTERLEAVED, patch_frame=W.CANONICAL_FRAME),
    "gqa_rank0": lambda: W.gqa_video(num_layers=2, n_chunks=2, T=33, rank=0, page_size=16),
    "mla_rank8": lambda: W.mla_lite(num_layers=2, n_chunks=2, T=40, rank=8, page_size=16),
    "tiny_mha": W.tiny_mha,
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_operator_matches_independent_formulation(oracle_lib, case):
    wl = CASES[case]()
    err, pk, pv, wk, wv = _run_oracle(wl)
    assert err == 0
    ik, iv, iwk, iwv = _independent_reuse(wl)
    np.testing.assert_array_equal(wk.astype(bool), iwk)
    np.testing.assert_allclose(pk[iwk], ik[iwk], rtol=0, atol=1e-10)
    # untouched slots keep their input bits (sentinel NaN here)
    assert np.isnan(pk[~iwk]).all()
    if wl.n_ch == 2:
        np.testing.assert_array_equal(wv.astype(bool), iwv)
        np.testing.assert_allclose(pv[iwv], iv[iwv], rtol=0, atol=1e-10)


def test_rank0_and_mla_ckv_are_exact_copies(oracle_lib):
    """m = 0 is pure relocation; MLA c_KV is reused byte for byte."""
    wl = W.mla_lite(num_layers=2, n_chunks=2, T=40, rank=0, page_size=16)
    err, pk, _, wk, _ = _run_oracle(wl)
    assert err == 0
    for it in wl.items:
        pos = int(it["dst_pos"]) + np.arange(int(it["n_tokens"]))
        pages = wl.block_table[0, pos // 16]
        for layer in range(2):
            src = _bits_to_f64(wl.store_rows(int(it["chunk_id"]), layer, 0))
            np.testing.assert_array_equal(pk[layer, pages, pos % 16, :512], src[:, :512])


def test_delta_zero_rank_zero_is_bitwise_copy(oracle_lib):
    wl = W.gqa_video(num_layers=1, n_chunks=2, T=20, rank=0, page_size=16)
    wl.items["delta"] = 0
    err, pk, pv, wk, wv = _run_oracle(wl)
    for it in wl.items:
        pos = int(it["dst_pos"]) + np.arange(int(it["n_tokens"]))
        pages = wl.block_table[0, pos // 16]
        for ch, img in ((0, pk), (1, pv)):
            np.testing.assert_array_equal(img[0, pages, pos % 16], _bits_to_f64(wl.store_rows(int(it["chunk_id"]), 0, ch)))


def test_sliding_window_in_place_rotates_keys_only(oracle_lib):
    """Kamera §3 sliding-window survival: survivors need only R(delta), V and
    the evicted pages are untouched."""
    wl = W.sliding_window(num_layers=2, n_resident=6, n_evict=2, T=32, page_size=16, num_kv_heads=2)
    k_in, v_in = wl.host_pool(0), wl.host_pool(1)
    err, pk, pv, wk, wv = _run_oracle(wl, k_in, v_in)
    assert err == 0
    np.testing.assert_array_equal(pv, _bits_to_f64(v_in))
    assert not wv.any()
    theta = _theta_np(wl.rope_base, 128)
    kin = _bits_to_f64(k_in)
    surv_pages = set(wl.block_table[0].tolist())
    for layer in range(2):
        for page in range(wl.num_pages):
            if page in surv_pages:
                want = _complex_rotate_rows(kin[layer, page], 2, 128, 128, 0, -64, theta, W.ROTATE_HALF)
                np.testing.assert_allclose(pk[layer, page], want, atol=1e-10)
                assert wk[layer, page].all()
            else:
                np.testing.assert_array_equal(pk[layer, page], kin[layer, page])


def test_apply_patch_in_place_adds_without_rotation(oracle_lib):
    wl = _small_gqa().replace(mode="apply_patch", pool_init="random", chunk_lens=[])
    k_in, v_in = wl.host_pool(0), wl.host_pool(1)
    err, pk, pv, wk, wv = _run_oracle(wl, k_in, v_in)
    assert err == 0
    it = wl.items[1]
    pos = int(it["dst_pos"]) + np.arange(int(it["n_tokens"]))
    pages, slots = wl.block_table[0, pos // 16], pos % 16
    for ch, img, src in ((0, pk, k_in), (1, pv, v_in)):
        U = _bits_to_f64(wl.u_rows(1, 1, ch))
        V = _bits_to_f64(wl.v_rows(1, 1, ch))
        want = _bits_to_f64(src[1, pages, slots]) + U @ V.T
        np.testing.assert_allclose(img[1, pages, slots], want, atol=1e-12)


def test_error_bits_and_skips(oracle_lib):
    wl = _small_gqa()
    items = wl.items.copy()
    items[0]["chunk_id"] = 99        # chunk out of range -> whole item skipped
    items[1]["patch_id"] = 42        # patch out of range -> skipped
    items[2]["dst_pos"] = 3 * 70 - 5  # runs past the block table -> its last rows skipped
    wl2 = wl.replace(items=items)
    err, pk, pv, wk, wv = _run_oracle(wl2)
    assert err == (oracle.EFLAG_CHUNK_OOB | oracle.EFLAG_PATCH_OOB | oracle.EFLAG_PAGE_OOB)
    n_pos = wl.block_table.shape[1] * 16
    expect_rows = 2 * (n_pos - (3 * 70 - 5))
    assert int(wk.sum()) == expect_rows and int(wv.sum()) == expect_rows
    items = wl.items.copy()
    items[0]["n_tokens"] = 69        # length disagrees with the store
    err, *_ = _run_oracle(wl.replace(items=items))
    assert err == oracle.EFLAG_LEN


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_workloads_match_independent_formulation(oracle_lib, seed):
    """The seeded random batches of the GPU fuzz (family, head size, partial
    rotary, rank, page size, pairing, frame, M-RoPE sections, ragged chunks
    reused at several positions, several sequences, patched and unpatched
    items) through the oracle and through the independent formulation."""
    from tests.harness import oracle_reference
    from tests.test_gpu_fuzz import random_workload

    wl = random_workload(1000 + seed)
    err, pk, pv, wk, wv = oracle_reference(wl)
    assert err == 0
    ik, iv, iwk, iwv = _independent_reuse(wl)
    np.testing.assert_array_equal(wk.astype(bool), iwk)
    np.testing.assert_allclose(pk[iwk], ik[iwk], rtol=0, atol=1e-9)
    np.testing.assert_array_equal(pk[~iwk], ik[~iwk])
    if wl.n_ch == 2:
        np.testing.assert_array_equal(wv.astype(bool), iwv)
        np.testing.assert_allclose(pv[iwv], iv[iwv], rtol=0, atol=1e-9)
        np.testing.assert_array_equal(pv[~iwv], iv[~iwv])


def _independent_in_place(wl, pool_k, pool_v):
    """The in-place modes as matrix algebra: relocation turns the K rows at
    each item's slots by its shift (V untouched); the patch mode adds U V^T to
    the K and V rows at the slots of each patched item, with no rotation."""
    theta = _theta_np(wl.rope_base, wl.rope_dim)
    pk = _bits_to_f64(pool_k)
    pv = _bits_to_f64(pool_v) if pool_v is not None else None
    wk = np.zeros(pk.shape[:-1], bool)
    wv = np.zeros(pk.shape[:-1], bool)
    for i_it, it in enumerate(wl.items):
        T, p, delta = int(it["n_tokens"]), int(it["patch_id"]), int(it["delta"])
        if sum(wl.rope_sections) and wl.section_deltas is not None:
            delta = np.repeat(np.asarray(wl.section_deltas[i_it], np.float64), wl.rope_sections)
        pos = int(it["dst_pos"]) + np.arange(T)
        pages, slots = wl.block_table[int(it["seq"]), pos // wl.page_size], pos % wl.page_size
        for layer in range(wl.num_layers):
            if wl.mode == "relocate_in_place":
                if wl.family == W.MLA:
                    heads, stride, col0 = 1, 0, wl.latent_dim
                else:
                    heads, stride, col0 = wl.num_kv_heads, wl.head_dim, 0
                x = pk[layer, pages, slots]
                pk[layer, pages, slots] = _complex_rotate_rows(x, heads, wl.rope_dim, stride, col0, delta, theta,
                                                               wl.pairing)
                wk[layer, pages, slots] = True
            elif p >= 0:
                for ch in range(wl.n_ch):
                    img, w = (pk, wk) if ch == 0 else (pv, wv)
                    U = _bits_to_f64(wl.u_rows(p, layer, ch))
                    V = _bits_to_f64(wl.v_rows(p, layer, ch))
                    img[layer, pages, slots] = img[layer, pages, slots] + U @ V.T
                    w[layer, pages, slots] = True
    return pk, pv, wk, wv


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_in_place_modes_match_independent_formulation(oracle_lib, seed):
    """The seeded random batches of the GPU fuzz of the in-place modes
    (sliding-window relocation for even seeds, patch in place for odd ones)
    through the oracle and through the independent formulation."""
    from tests.harness import oracle_reference
    from tests.test_gpu_fuzz import random_workload

    base = random_workload(2000 + seed)
    mode = "relocate_in_place" if seed % 2 == 0 else "apply_patch"
    if mode == "apply_patch" and base.rank == 0:
        base = base.replace(rank=16, patch_lens=base.chunk_lens)
        base.items["patch_id"] = base.items["chunk_id"]
    wl = base.replace(mode=mode, pool_init="random")
    if mode == "apply_patch":
        _, first = np.unique(wl.items["chunk_id"], return_index=True)
        wl = wl.replace(items=wl.items[np.sort(first)].copy())
    pool_k, pool_v = wl.host_pool(0), wl.host_pool(1) if wl.n_ch == 2 else None
    err, pk, pv, wk, wv = oracle_reference(wl, pool_k, pool_v)
    assert err == 0
    ik, iv, iwk, iwv = _independent_in_place(wl, pool_k, pool_v)
    np.testing.assert_array_equal(wk.astype(bool), iwk)
    np.testing.assert_allclose(pk[iwk], ik[iwk], rtol=0, atol=1e-9)
    np.testing.assert_array_equal(pk[~iwk], ik[~iwk])
    if wl.n_ch == 2:
        np.testing.assert_array_equal(wv.astype(bool), iwv)
        np.testing.assert_allclose(pv[iwv], iv[iwv], rtol=0, atol=1e-9)
        np.testing.assert_array_equal(pv[~iwv], iv[~iwv])
