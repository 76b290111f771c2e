"""Seeded fuzz of the CUDA path against the fp64 oracle: random family, head
dimension, rank, page size, pairing, patch frame, ragged lengths, chunks
reused at several positions, items sharing pages at disjoint slots, patched
and unpatched items mixed in one batch, several sequences."""
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
    torch.cuda.set_device(0)


def random_workload(seed: int, compressed: bool = False) -> W.Workload:
    """compressed: shapes the compressed store serves (MHA/GQA, head_dim 64 or
    128, D a multiple of 128)."""
    rng = np.random.default_rng(seed)
    family = int(rng.choice([W.MHA, W.GQA] if compressed else [W.MHA, W.GQA, W.MLA]))
    kw = {}
    if family == W.MLA:
        kw.update(latent_dim=int(rng.choice([128, 256, 512])), rope_dim=64)
    else:
        hd = int(rng.choice([64, 128] if compressed else [64, 128, 256]))
        heads = int(rng.integers(1, max(2, min(5, 1024 // hd + 1))))
        if compressed and hd == 64 and heads % 2:
            heads += 1
        rope = hd if rng.random() < 0.7 or hd == 64 else 64
        kw.update(num_kv_heads=heads, head_dim=hd, rope_dim=rope)
    L = int(rng.integers(1, 4))
    n_chunks = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.choice([1, 7, 63, 64, 65, 127, 128, 129, 300], n_chunks)]
    rank = int(rng.choice([0, 8, 16, 32, 64]))
    P = int(rng.choice([8, 16, 64, 128, 256]))
    n_seqs = int(rng.integers(1, 3))
    # items: every chunk once, some twice, placed with random gaps per sequence
    uses = list(range(n_chunks)) + [int(c) for c in rng.integers(0, n_chunks, int(rng.integers(0, 3)))]
    rng.shuffle(uses)
    cursor = [0] * n_seqs
    rows = []
    for c in uses:
        sq = int(rng.integers(0, n_seqs))
        cursor[sq] += int(rng.integers(0, P + 1))
        pid = c if (rank and rng.random() < 0.75) else -1
        delta = int(rng.integers(-70000, 70000))
        rows.append((c, pid, delta, sq, lens[c], cursor[sq]))
        cursor[sq] += lens[c]
    items = W.make_items(*[np.array(col) for col in zip(*rows)])
    ppseq = max(1, -(-max(cursor) // P))
    num_pages = n_seqs * ppseq + int(rng.integers(0, 4))
    bt = W.shuffled_block_table(seed, n_seqs, ppseq, num_pages)
    mrope = {}
    if rng.random() < 0.3:
        npairs = (kw.get("rope_dim") or 64) // 2
        a = int(rng.integers(0, npairs + 1))
        b = int(rng.integers(0, npairs - a + 1))
        sec = (a, b, npairs - a - b)
        mrope = dict(rope_sections=sec,
                     section_deltas=rng.integers(-70000, 70000, (len(items), 3)).astype(np.int64))
    return W.Workload(f"fuzz{seed}", family, L, rope_base=float(rng.choice([1e4, 5e5, 1e6])), **mrope,
                      pairing=int(rng.integers(0, 2)), patch_frame=int(rng.integers(0, 2)), chunk_lens=lens,
                      rank=rank, patch_lens=lens if rank else [], items=items, page_size=P, num_pages=num_pages,
                      block_table=bt, seed=seed, sigma_uv=float(rng.choice([0.02, 0.3])), **kw)


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_reuse(seed):
    wl = random_workload(1000 + seed)
    t = H.device_inputs(wl, torch)
    H.call(wl, t)
    torch.cuda.synchronize()
    err, ref_k, ref_v, wk, wv = H.oracle_reference(wl)
    assert int(t["err"].item()) == err
    exact = slice(0, wl.latent_dim) if (wl.family == W.MLA and wl.rank == 0) else None
    H.assert_report(H.compare_pool(H.to_bits(t["pool_k"]), wl.host_pool(0), ref_k, wk, exact))
    if wl.n_ch == 2:
        H.assert_report(H.compare_pool(H.to_bits(t["pool_v"]), wl.host_pool(1), ref_v, wv))


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_in_place_modes(seed):
    base = random_workload(2000 + seed)
    mode = "relocate_in_place" if seed % 2 == 0 else "apply_patch"
    if mode == "apply_patch" and base.rank == 0:
        base = base.replace(rank=16, patch_lens=base.chunk_lens)
        base.items["patch_id"] = base.items["chunk_id"]
    wl = base.replace(mode=mode, pool_init="random")
    if mode == "apply_patch":
        # in place, two items must not share a slot: keep one use per chunk
        _, first = np.unique(wl.items["chunk_id"], return_index=True)
        wl = wl.replace(items=wl.items[np.sort(first)].copy())
    pool = (wl.host_pool(0), wl.host_pool(1) if wl.n_ch == 2 else None)
    t = H.device_inputs(wl, torch, pool_host=pool)
    H.call(wl, t)
    torch.cuda.synchronize()
    err, ref_k, ref_v, wk, wv = H.oracle_reference(wl, pool[0], pool[1])
    assert int(t["err"].item()) == err
    exact = slice(0, wl.latent_dim) if wl.family == W.MLA and mode == "relocate_in_place" else None
    H.assert_report(H.compare_pool(H.to_bits(t["pool_k"]), pool[0], ref_k, wk, exact))
    if wl.n_ch == 2:
        H.assert_report(H.compare_pool(H.to_bits(t["pool_v"]), pool[1], ref_v, wv))


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_compressed_store(seed):
    """kamera_reuse_compressed on random shapes; the store is the oracle's
    encoding of the bf16 store (even seeds) or seeded random contents (odd)."""
    import oracle

    wl = random_workload(3000 + seed, compressed=True)
    if seed % 2 == 0:
        m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim)
        arrs = H.comp_arrays(oracle.compress_store(m, wl.host_store(), wl.store_off,
                                                   np.array(wl.chunk_lens, np.int32),
                                                   row_offset=wl.comp_row_offset, n_rows=wl.comp_rows))
    else:
        arrs = H.comp_arrays(wl.random_compressed())
    cstore, _ct = H.device_compressed(arrs, torch)
    t = H.device_inputs(wl, torch, with_store=False)
    H.call_compressed(wl, t, cstore)
    torch.cuda.synchronize()
    err, ref_k, ref_v, wk, wv = H.oracle_reference_compressed(wl, H.oracle_store(arrs))
    assert int(t["err"].item()) == err
    H.assert_report(H.compare_pool(H.to_bits(t["pool_k"]), wl.host_pool(0), ref_k, wk))
    H.assert_report(H.compare_pool(H.to_bits(t["pool_v"]), wl.host_pool(1), ref_v, wv))
