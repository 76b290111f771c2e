"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, on seeded workloads that span several tiles and ragged
tails, for every family, window operation, rank and pairing.

Kamera §2 reuse equation, relocation and patch application; §3 window
operations.  Tolerance: one bf16 ulp of the oracle value + 1e-3 on rotated or
patched values; bit-exact for untouched slots, unpatched c_KV and copies.
"""
import numpy as np
import pytest

from synth import workloads as W
from tests import harness as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import position_invariant_kv_kamera_gb300 as pk

    pk.load()
    torch.cuda.set_device(0)


def run_and_compare(wl, exact_k_cols=None, mode=None, pool_host=None):
    pool_k_in = pool_host[0] if pool_host else wl.host_pool(0)
    pool_v_in = (pool_host[1] if pool_host else wl.host_pool(1)) if wl.n_ch == 2 else None
    t = H.device_inputs(wl, torch, pool_host=(pool_k_in, pool_v_in) if pool_host else None)
    H.call(wl, t, mode=mode)
    torch.cuda.synchronize()
    err, ref_k, ref_v, wk, wv = H.oracle_reference(wl, pool_k_in, pool_v_in)
    assert int(t["err"].item()) == err
    rep_k = H.compare_pool(H.to_bits(t["pool_k"]), pool_k_in, ref_k, wk, exact_k_cols)
    H.assert_report(rep_k)
    reps = [rep_k]
    if wl.n_ch == 2:
        rep_v = H.compare_pool(H.to_bits(t["pool_v"]), pool_v_in, ref_v, wv)
        H.assert_report(rep_v)
        reps.append(rep_v)
    return reps, t


def test_generator_device_twin_is_bit_identical():
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=300, rank=32)
    t = H.device_inputs(wl, torch)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(H.to_bits(t["store"]), wl.host_store())
    np.testing.assert_array_equal(H.to_bits(t["patch"]), wl.host_patch())
    sw = W.sliding_window(num_layers=2, n_resident=3, n_evict=1, T=64, page_size=16, num_kv_heads=2)
    np.testing.assert_array_equal(H.to_bits(sw.device_pool(torch, 1)), sw.host_pool(1))


def test_tiny_mha_contiguous_output():
    """MHA, 1 layer, 4 x 64, T = 256, rank 8, delta 1000, base 1e4, rotate-half,
    into a contiguous [256][4][64] buffer."""
    reps, _ = run_and_compare(W.tiny_mha())
    assert reps[0]["rows_written"] == 256


@pytest.mark.parametrize("rank", [0, 8, 16, 32, 64])
@pytest.mark.parametrize("page_size", [16, 64])
def test_gqa_ranks_and_pages(rank, page_size):
    wl = W.gqa_video(num_layers=2, n_chunks=3, T=300, rank=rank, page_size=page_size)
    # shift the chunks so they start mid-page and leave gaps between them
    wl.items["dst_pos"] = np.array([5, 333, 700])
    wl.block_table = W.shuffled_block_table(wl.seed, 1, -(-1000 // page_size))
    wl.num_pages = wl.block_table.shape[1]
    run_and_compare(wl)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 129, 1296])
def test_ragged_chunk_lengths(T):
    wl = W.gqa_video(num_layers=1, n_chunks=2, T=T, rank=16, page_size=64)
    run_and_compare(wl)


def test_gqa_interleaved_canonical_frame():
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=200, rank=32).replace(pairing=W.INTERLEAVED,
                                                                         patch_frame=W.CANONICAL_FRAME)
    run_and_compare(wl)


def test_gqa_relocate_through_store_matches_reuse_without_patch():
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=150, rank=0)
    run_and_compare(wl, mode="relocate")


@pytest.mark.parametrize("rank", [0, 8, 16])
def test_mla(rank):
    wl = W.mla_lite(num_layers=2, n_chunks=3, T=300, rank=rank, page_size=64)
    wl.items["dst_pos"] = np.array([0, 301, 640])
    wl.block_table = W.shuffled_block_table(wl.seed, 1, -(-940 // 64))
    wl.num_pages = wl.block_table.shape[1]
    run_and_compare(wl, exact_k_cols=slice(0, 512) if rank == 0 else None)


def test_sliding_window_in_place():
    wl = W.sliding_window(num_layers=2, n_resident=6, n_evict=2, T=256, page_size=64, num_kv_heads=4)
    pool = (wl.host_pool(0), wl.host_pool(1))
    reps, t = run_and_compare(wl, pool_host=pool)
    # V is not touched at all
    np.testing.assert_array_equal(H.to_bits(t["pool_v"]), pool[1])


def test_mla_in_place_relocation_keeps_ckv_bits():
    wl = W.mla_lite(num_layers=2, n_chunks=2, T=200, rank=0, page_size=16).replace(
        mode="relocate_in_place", chunk_lens=[], pool_init="random")
    run_and_compare(wl, exact_k_cols=slice(0, 512), pool_host=(wl.host_pool(0), None))


def test_apply_patch_in_place():
    wl = W.gqa_video(num_layers=2, n_chunks=3, T=200, rank=32, page_size=16).replace(
        mode="apply_patch", chunk_lens=[], pool_init="random")
    run_and_compare(wl, pool_host=(wl.host_pool(0), wl.host_pool(1)))


def test_long_video_reorder_and_recall_small():
    wl = W.long_video(num_layers=2, n_reorder=6, n_recall=2, T=1296, rank=64)
    run_and_compare(wl)


def test_delta_zero_rank_zero_is_a_bitwise_copy():
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=100, rank=0, page_size=16)
    wl.items["delta"] = 0
    _, t = run_and_compare(wl)
    k = H.to_bits(t["pool_k"])
    for it in wl.items:
        pos = int(it["dst_pos"]) + np.arange(int(it["n_tokens"]))
        pages = wl.block_table[0, pos // 16]
        for layer in range(2):
            np.testing.assert_array_equal(k[layer, pages, pos % 16], wl.store_rows(int(it["chunk_id"]), layer, 0))


def test_zero_patch_equals_relocation_bitwise():
    wl = W.gqa_video(num_layers=1, n_chunks=2, T=100, rank=16, page_size=16).replace(sigma_uv=0.0)
    t = H.device_inputs(wl, torch)
    H.call(wl, t)
    t0 = H.device_inputs(wl.replace(rank=0, patch_lens=[]), torch)
    H.call(wl.replace(rank=0, patch_lens=[]), t0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(H.to_bits(t["pool_k"]), H.to_bits(t0["pool_k"]))
    np.testing.assert_array_equal(H.to_bits(t["pool_v"]), H.to_bits(t0["pool_v"]))


def test_stress_patch_scale():
    """Patches of O(1) size (U, V ~ N(0, 0.3)) exercise the tolerance."""
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=257, rank=64).replace(sigma_uv=0.3)
    run_and_compare(wl)


def test_error_flags_and_skips():
    wl = W.gqa_video(num_layers=2, n_chunks=4, T=70, rank=16, page_size=16)
    items = wl.items.copy()
    items[0]["chunk_id"] = 99
    items[1]["patch_id"] = 42
    items[3]["dst_pos"] = 4 * 70 - 5
    wl = wl.replace(items=items)
    run_and_compare(wl)
    items = wl.items.copy()
    items[0]["n_tokens"] = 69
    items[1]["seq"] = 3
    items[2]["dst_pos"] = -1
    run_and_compare(wl.replace(items=items))


@pytest.mark.parametrize("pairing", [W.ROTATE_HALF, W.INTERLEAVED])
@pytest.mark.parametrize("rank", [0, 32])
def test_mrope_sections(pairing, rank):
    """M-RoPE (temporal / height / width sections of 16 / 24 / 24 pairs): each
    section re-rotated by its own shift."""
    wl = W.with_mrope(W.gqa_video(num_layers=2, n_chunks=3, T=200, rank=rank, page_size=16)).replace(
        pairing=pairing)
    if rank == 0:
        wl = wl.replace(patch_lens=[])
    run_and_compare(wl)


def test_mrope_in_place_sliding_window():
    wl = W.with_mrope(W.sliding_window(num_layers=2, n_resident=4, n_evict=1, T=128, page_size=64,
                                       num_kv_heads=2))
    run_and_compare(wl, pool_host=(wl.host_pool(0), wl.host_pool(1)))


def test_mrope_equal_section_shifts_match_plain_rope_bitwise():
    base = W.gqa_video(num_layers=1, n_chunks=2, T=150, rank=16, page_size=16)
    sd = np.repeat(base.items["delta"][:, None], 3, axis=1)
    wl = base.replace(rope_sections=(16, 24, 24), section_deltas=sd)
    t0 = H.device_inputs(base, torch)
    H.call(base, t0)
    t1 = H.device_inputs(wl, torch)
    H.call(wl, t1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(H.to_bits(t0["pool_k"]), H.to_bits(t1["pool_k"]))


def scaled_inv_freq(base: float, rope_dim: int, factor: float = 8.0, ctx: float = 8192.0, lo: float = 1.0,
                    hi: float = 4.0) -> np.ndarray:
    """A long-context scaled frequency table (the frequency-dependent scaling
    of Llama 3.1's RoPE): pairs whose wavelength 2 pi / theta is longer than
    ctx / lo turn `factor` times slower, pairs shorter than ctx / hi keep their
    frequency, and the band between blends the two linearly in ctx / wavelength."""
    th = base ** (-2.0 * np.arange(rope_dim // 2) / rope_dim)
    wl = 2 * np.pi / th
    smooth = np.clip((ctx / wl - lo) / (hi - lo), 0.0, 1.0)
    return (1 - smooth) * th / factor + smooth * th


@pytest.mark.parametrize("family", [W.GQA, W.MLA])
@pytest.mark.parametrize("pairing", [W.ROTATE_HALF, W.INTERLEAVED])
def test_explicit_frequency_table(family, pairing):
    """R(delta) with an explicit frequency table (kamera_model_desc.inv_freq)
    in place of the base ladder: the same table drives the oracle."""
    if family == W.GQA:
        base = W.gqa_video(num_layers=2, n_chunks=3, T=200, rank=32, page_size=16)
    else:
        base = W.mla_lite(num_layers=2, n_chunks=2, T=150, rank=16, page_size=16)
    th = scaled_inv_freq(base.rope_base, base.rope_dim)
    assert not np.allclose(th, base.rope_base ** (-2.0 * np.arange(base.rope_dim // 2) / base.rope_dim))
    run_and_compare(base.replace(inv_freq=th, pairing=pairing))
