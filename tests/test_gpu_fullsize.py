"""Full-size parity: the five workload shapes at their real sizes (up to the
57 GB long-video reorder + recall), launched exactly as the benchmark
launches them, compared with the fp64 oracle on EVERY written row.

Layer by layer and channel by channel, the rows each item wrote are gathered
from the pool (destinations found by brute force on the block table), with
the canonical rows and patch factors they were computed from (the device
copies of the seeded generator's output, which the kernels read), and
``oracle.check_rows`` recomputes each row with the oracle's row function and
applies the comparison rule -- on all host cores, one item block per task.
Properties that hold at any size (which slots are written, sentinel slots
untouched, bit-exact copies) are checked over the whole pool on the device.
The compressed-store case decodes every row with the oracle's decoder
(``oracle.check_rows_compressed``)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests import harness as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

N_SAMPLES = 160


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _oracle_model(wl):
    return oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim, wl.latent_dim,
                        wl.pairing, wl.patch_frame, wl.rope_sections)


def _slot_rows(wl, item, t):
    """(page, slot) of token t of an item, by brute force on the block table."""
    pos = int(item["dst_pos"]) + t
    return int(wl.block_table[int(item["seq"]), pos // wl.page_size]), pos % wl.page_size


def _samples(wl, rng):
    out = []
    chans = 1 if wl.mode == "relocate_in_place" else wl.n_ch
    for _ in range(N_SAMPLES):
        i = int(rng.integers(0, len(wl.items)))
        it = wl.items[i]
        T = int(it["n_tokens"])
        # bias towards chunk edges (tile and page boundaries)
        t = int(rng.choice([0, T - 1, int(rng.integers(0, T)), min(T - 1, 127), min(T - 1, 128)]))
        out.append((i, int(rng.integers(0, wl.num_layers)), int(rng.integers(0, chans)), t))
    return out


def _dest_rows(wl, item) -> np.ndarray:
    """Pool rows (page * P + slot) of an item's tokens, by brute force on the block table."""
    pos = int(item["dst_pos"]) + np.arange(int(item["n_tokens"]))
    return (wl.block_table[int(item["seq"]), pos // wl.page_size].astype(np.int64) * wl.page_size
            + pos % wl.page_size)


def _gather(buf2d, rows: np.ndarray) -> np.ndarray:
    """Rows of a 2-D device tensor (any 16-bit dtype) as host uint16 bits."""
    idx = torch.from_numpy(rows).to(buf2d.device)
    return buf2d.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)


def _check_every_row(wl, t, fresh_pool=None):
    """Every row every item wrote, against the oracle; fresh_pool: the initial
    pool per channel (the in-place sources)."""
    m = _oracle_model(wl)
    th = H.oracle_theta(wl)
    L, D, P = wl.num_layers, wl.D, wl.page_size
    in_place = wl.mode == "relocate_in_place"
    chans = 1 if in_place else wl.n_ch
    patched = bool(wl.rank) and not in_place and "patch" in t
    rotate = wl.mode != "apply_patch"
    items = [it for it in wl.items if int(it["n_tokens"]) > 0]
    dst = [_dest_rows(wl, it) for it in items]
    bounds = np.cumsum([0] + [len(d) for d in dst])
    all_dst = np.concatenate(dst)
    deltas = [wl.section_deltas[i] if wl.section_deltas is not None else int(it["delta"])
              for i, it in enumerate(wl.items) if int(it["n_tokens"]) > 0]
    n_exact = wl.latent_dim if (wl.family == W.MLA and not patched) else 0
    store2d = t["store"].view(-1, D) if "store" in t else None
    patch2d = t["patch"].view(-1, wl.rank) if patched else None
    failures, rows_checked = [], 0
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        for layer in range(L):
            for ch in range(chans):
                pool = t["pool_k"] if ch == 0 else t["pool_v"]
                got = _gather(pool.view(L, -1, D)[layer], all_dst)
                if in_place:
                    src = _gather(fresh_pool[ch].view(L, -1, D)[layer], all_dst)
                else:
                    srows = np.concatenate([
                        int(wl.store_off[int(it["chunk_id"])]) // D
                        + (layer * wl.n_ch + ch) * int(it["n_tokens"]) + np.arange(int(it["n_tokens"]))
                        for it in items])
                    src = _gather(store2d, srows)
                u_all = v_all = None
                if patched:
                    urows, vrows = [], []
                    for it in items:
                        T = int(it["n_tokens"])
                        pid = int(it["patch_id"])
                        if pid < 0:
                            continue
                        base = int(wl.patch_off[pid]) // wl.rank + (layer * wl.n_ch + ch) * (T + D)
                        urows.append(base + np.arange(T))
                        vrows.append(base + T + np.arange(D))
                    u_all = _gather(patch2d, np.concatenate(urows)) if urows else None
                    v_all = _gather(patch2d, np.concatenate(vrows)) if vrows else None
                futs, ui, vi = [], 0, 0
                for k, it in enumerate(items):
                    a, b = bounds[k], bounds[k + 1]
                    u = v = None
                    if patched and int(it["patch_id"]) >= 0:
                        u = u_all[ui:ui + (b - a)]
                        v = v_all[vi:vi + D]
                        ui += b - a
                        vi += D
                    futs.append((k, ex.submit(oracle.check_rows, m, th, ch, deltas[k], src[a:b], got[a:b], u, v,
                                              rotate, n_exact if ch == 0 else 0)))
                for k, f in futs:
                    n_bad, max_err, first = f.result()
                    if n_bad:
                        failures.append((layer, ch, k, n_bad, max_err, divmod(first, D)))
                rows_checked += len(all_dst)
    assert not failures, (wl.name, failures[:10])
    assert rows_checked == len(all_dst) * L * chans


def _check_samples(wl, t, pool_init_rows=None):
    """Oracle rows for sampled (item, layer, channel, token) against the pool."""
    m = _oracle_model(wl)
    th = oracle.theta(wl.rope_base, wl.rope_dim)
    rng = np.random.default_rng(7)
    for (i, layer, ch, tok) in _samples(wl, rng):
        it = wl.items[i]
        page, slot = _slot_rows(wl, it, tok)
        if wl.mode == "relocate_in_place":
            src = pool_init_rows(ch, layer, page)[slot]
        else:
            src = wl.store_rows(int(it["chunk_id"]), layer, ch, tok, tok + 1)[0]
        u = v = None
        if wl.rank and int(it["patch_id"]) >= 0 and wl.mode != "relocate_in_place":
            u = H.bits_to_f64(wl.u_rows(int(it["patch_id"]), layer, ch, tok, tok + 1)[0])
            v = H.bits_to_f64(wl.v_rows(int(it["patch_id"]), layer, ch))
        delta = wl.section_deltas[i] if wl.section_deltas is not None else int(it["delta"])
        ref = oracle.row(m, th, ch, delta, H.bits_to_f64(src), u, v, rotate=wl.mode != "apply_patch")
        pool = t["pool_k"] if ch == 0 else t["pool_v"]
        got = H.to_bits(pool[layer, page, slot])
        ok = H.within_tol(H.bits_to_f64(got), ref)
        assert ok.all(), (wl.name, i, layer, ch, tok, np.abs(H.bits_to_f64(got) - ref).max())
        if wl.family == W.MLA and u is None:
            np.testing.assert_array_equal(got[:wl.latent_dim], src[:wl.latent_dim])


def _written_rows_mask(wl):
    """[num_pages * P] bool: slots that the items cover (same for every layer)."""
    mask = np.zeros(wl.num_pages * wl.page_size, bool)
    for it in wl.items:
        pos = int(it["dst_pos"]) + np.arange(int(it["n_tokens"]))
        pages = wl.block_table[int(it["seq"]), pos // wl.page_size]
        mask[pages * wl.page_size + pos % wl.page_size] = True
    return mask


def _check_sentinel_coverage(wl, pool):
    """Every covered slot fully written (no NaN sentinel left), every other
    slot still all-sentinel."""
    bits = pool.view(torch.int16).reshape(wl.num_layers, -1, wl.D)
    any_sent = (bits == -1).any(dim=-1)
    all_sent = (bits == -1).all(dim=-1)
    mask = torch.from_numpy(_written_rows_mask(wl)).to(pool.device)
    assert not any_sent[:, mask].any().item(), "a covered slot was not (fully) written"
    assert all_sent[:, ~mask].all().item(), "an uncovered slot was written"


def _gather_rows(wl, pool, item):
    pos = int(item["dst_pos"]) + np.arange(int(item["n_tokens"]))
    rows = wl.block_table[int(item["seq"]), pos // wl.page_size] * wl.page_size + pos % wl.page_size
    idx = torch.from_numpy(rows.astype(np.int64)).to(pool.device)
    return pool.reshape(wl.num_layers, -1, wl.D)[:, idx]


def _run(wl):
    t = H.device_inputs(wl, torch)
    H.call(wl, t)
    torch.cuda.synchronize()
    assert int(t["err"].item()) == 0
    return t


def test_full_tiny_mha():
    wl = W.tiny_mha()
    t = _run(wl)
    _check_sentinel_coverage(wl, t["pool_k"])
    _check_sentinel_coverage(wl, t["pool_v"])
    _check_every_row(wl, t)
    _check_samples(wl, t)


def test_full_gqa_video():
    wl = W.gqa_video()
    t = _run(wl)
    _check_sentinel_coverage(wl, t["pool_k"])
    _check_sentinel_coverage(wl, t["pool_v"])
    _check_every_row(wl, t)
    _check_samples(wl, t)


def test_full_gqa_video_mrope():
    """The headline shape with multimodal RoPE sections (16/24/24 pairs) and
    separate temporal and spatial shifts per chunk."""
    wl = W.with_mrope(W.gqa_video())
    t = _run(wl)
    _check_sentinel_coverage(wl, t["pool_k"])
    _check_every_row(wl, t)
    _check_samples(wl, t)


@pytest.mark.parametrize("rank", [16, 0])
def test_full_mla_lite(rank):
    wl = W.mla_lite(rank=rank)
    t = _run(wl)
    _check_sentinel_coverage(wl, t["pool_k"])
    _check_every_row(wl, t)  # rank 0: c_KV columns bit-exact on every row
    _check_samples(wl, t)
    if rank == 0:
        # c_KV byte for byte, over every reused row of every layer
        store = t["store"]
        for it in wl.items:
            c = int(it["chunk_id"])
            T = int(it["n_tokens"])
            src = store[int(wl.store_off[c]):int(wl.store_off[c]) + wl.num_layers * T * wl.D]
            src = src.view(torch.int16).reshape(wl.num_layers, T, wl.D)[..., :wl.latent_dim]
            got = _gather_rows(wl, t["pool_k"], it).view(torch.int16)[..., :wl.latent_dim]
            assert torch.equal(src, got)


def test_full_sliding_window():
    wl = W.sliding_window()
    t = _run(wl)
    # V untouched, K of evicted pages untouched: compare with a fresh fill
    assert torch.equal(t["pool_v"].view(torch.int16), wl.device_pool(torch, 1).view(torch.int16))
    fresh_k = wl.device_pool(torch, 0)
    surv = torch.from_numpy(np.unique(wl.block_table[0]).astype(np.int64)).cuda()
    evicted = torch.ones(wl.num_pages, dtype=torch.bool, device="cuda")
    evicted[surv] = False
    assert torch.equal(t["pool_k"][:, evicted].view(torch.int16), fresh_k[:, evicted].view(torch.int16))
    _check_every_row(wl, t, fresh_pool=[fresh_k])
    del fresh_k
    _check_samples(wl, t, pool_init_rows=wl.pool_rows)


def test_full_long_video():
    wl = W.long_video()
    t = _run(wl)
    _check_sentinel_coverage(wl, t["pool_k"])
    _check_sentinel_coverage(wl, t["pool_v"])
    _check_every_row(wl, t)
    _check_samples(wl, t)
    del t
    torch.cuda.empty_cache()


def _check_every_row_compressed(wl, t, ocs):
    """Every row every item wrote from the compressed store, against the oracle
    (decode, rotate, patch), layer by layer and item block by item block on all
    host cores."""
    m = _oracle_model(wl)
    th = H.oracle_theta(wl)
    L, D = wl.num_layers, wl.D
    items = [it for it in wl.items if int(it["n_tokens"]) > 0]
    dst = [_dest_rows(wl, it) for it in items]
    bounds = np.cumsum([0] + [len(d) for d in dst])
    all_dst = np.concatenate(dst)
    patch2d = t["patch"].view(-1, wl.rank)
    failures = []
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        for layer in range(L):
            for ch in range(2):
                pool = t["pool_k"] if ch == 0 else t["pool_v"]
                got = _gather(pool.view(L, -1, D)[layer], all_dst)
                futs = []
                for k, it in enumerate(items):
                    T, pid = int(it["n_tokens"]), int(it["patch_id"])
                    base = int(wl.patch_off[pid]) // wl.rank + (layer * 2 + ch) * (T + D)
                    u = _gather(patch2d, base + np.arange(T))
                    v = _gather(patch2d, base + T + np.arange(D))
                    futs.append((k, ex.submit(oracle.check_rows_compressed, m, th, ocs, int(it["chunk_id"]), layer, ch,
                                              0, int(it["delta"]), got[bounds[k]:bounds[k + 1]], u, v)))
                for k, f in futs:
                    n_bad, max_err, first = f.result()
                    if n_bad:
                        failures.append((layer, ch, k, n_bad, max_err, divmod(first, D)))
    assert not failures, failures[:10]


def test_full_gqa_video_compressed():
    """The headline batch reused from a compressed store at full size (458,752
    store rows, 0.33 GB of codes) in the bench's launch configuration, with
    seeded random contents: every written row is decoded and recomputed by the
    oracle, and sampled rows once more from host-regenerated patch factors."""
    wl = W.gqa_video()
    arrs = H.comp_arrays(wl.random_compressed())
    cstore, _ct = H.device_compressed(arrs, torch)
    t = H.device_inputs(wl, torch, with_store=False)
    H.call_compressed(wl, t, cstore)
    torch.cuda.synchronize()
    assert int(t["err"].item()) == 0
    _check_sentinel_coverage(wl, t["pool_k"])
    _check_sentinel_coverage(wl, t["pool_v"])
    m = _oracle_model(wl)
    th = oracle.theta(wl.rope_base, wl.rope_dim)
    ocs = H.oracle_store(arrs)
    rng = np.random.default_rng(11)
    for (i, layer, ch, tok) in _samples(wl, rng):
        it = wl.items[i]
        page, slot = _slot_rows(wl, it, tok)
        src = oracle.decode_row(m, ocs, int(it["chunk_id"]), layer, ch, tok)
        u = H.bits_to_f64(wl.u_rows(int(it["patch_id"]), layer, ch, tok, tok + 1)[0])
        v = H.bits_to_f64(wl.v_rows(int(it["patch_id"]), layer, ch))
        ref = oracle.row(m, th, ch, int(it["delta"]), src, u, v)
        got = H.to_bits((t["pool_k"] if ch == 0 else t["pool_v"])[layer, page, slot])
        ok = H.within_tol(H.bits_to_f64(got), ref)
        assert ok.all(), (i, layer, ch, tok, np.abs(H.bits_to_f64(got) - ref).max())
    _check_every_row_compressed(wl, t, ocs)
