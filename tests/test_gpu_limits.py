"""The CUDA path at the edges of what the library serves, against the fp64
oracle: the widest row (D = 2048, the largest head_dim 256, a 1984 + 64 MLA
latent row), the largest rank (64), pages far larger than a chunk, a single
long chunk; patch formation at the largest slab (8192 x 2048, k = 96) and on
degenerate slabs smaller than k.  Tolerances as in the other parity tests."""
import numpy as np
import pytest

from synth import gen
from synth import workloads as W
from tests import harness as H
from tests.test_gpu_factor import assert_product_matches

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def run_and_compare(wl):
    t = H.device_inputs(wl, torch)
    H.call(wl, t)
    torch.cuda.synchronize()
    err, ref_k, ref_v, wk, wv = H.oracle_reference(wl)
    assert int(t["err"].item()) == err == 0
    H.assert_report(H.compare_pool(H.to_bits(t["pool_k"]), wl.host_pool(0), ref_k, wk))
    if wl.n_ch == 2:
        H.assert_report(H.compare_pool(H.to_bits(t["pool_v"]), wl.host_pool(1), ref_v, wv))


def test_widest_gqa_row_rank_64():
    """16 KV heads x 128 = 2048 columns (the largest D), rank 64, 16-slot pages."""
    wl = W.gqa_video(num_layers=1, n_chunks=2, T=200, rank=64, page_size=16).replace(num_kv_heads=16)
    run_and_compare(wl)


def test_largest_head_dim_interleaved():
    """MHA with head_dim 256 (the largest served), 8 heads (D = 2048), interleaved pairs."""
    wl = W.gqa_video(num_layers=1, n_chunks=2, T=150, rank=32, page_size=64).replace(
        family=W.MHA, num_kv_heads=8, head_dim=256, rope_dim=256, pairing=W.INTERLEAVED)
    run_and_compare(wl)


def test_widest_mla_latent():
    """MLA latent row of 1984 + 64 = 2048 columns, rank 16."""
    wl = W.mla_lite(num_layers=1, n_chunks=2, T=130, rank=16).replace(latent_dim=1984)
    run_and_compare(wl)


def test_page_larger_than_the_chunks():
    """2048-slot pages: every chunk lands inside one page, at odd offsets."""
    wl = W.gqa_video(num_layers=2, n_chunks=3, T=300, rank=16, page_size=2048)
    wl.items["dst_pos"] = np.array([3, 400, 1500])
    wl.block_table = W.shuffled_block_table(wl.seed, 1, 1, 2)
    wl.num_pages = 2
    run_and_compare(wl)


def test_one_long_chunk():
    """A single 5000-token chunk (40 row blocks) starting mid-page."""
    wl = W.gqa_video(num_layers=1, n_chunks=1, T=5000, rank=32, page_size=64)
    wl.items["dst_pos"] = np.array([37])
    wl.block_table = W.shuffled_block_table(wl.seed, 1, -(-5037 // 64))
    wl.num_pages = wl.block_table.shape[1]
    run_and_compare(wl)


def test_compressed_store_widest_row():
    """The compressed store at D = 2048 (16 heads x 128), rank 64."""
    wl = W.gqa_video(num_layers=1, n_chunks=2, T=200, rank=64, page_size=16).replace(num_kv_heads=16)
    arrs = H.comp_arrays(wl.random_compressed())
    cstore, _ct = H.device_compressed(arrs, torch)
    t = H.device_inputs(wl, torch, with_store=False)
    H.call_compressed(wl, t, cstore)
    torch.cuda.synchronize()
    err, ref_k, ref_v, wk, wv = H.oracle_reference_compressed(wl, H.oracle_store(arrs))
    assert int(t["err"].item()) == err == 0
    H.assert_report(H.compare_pool(H.to_bits(t["pool_k"]), wl.host_pool(0), ref_k, wk))
    H.assert_report(H.compare_pool(H.to_bits(t["pool_v"]), wl.host_pool(1), ref_v, wv))


# ---- patch formation at its limits --------------------------------------------------------------

def _factor(deltas, m, p, q, seed=9):
    import position_invariant_kv_kamera_gb300 as pk

    n, T, D = deltas.shape
    d_dev = torch.from_numpy(np.ascontiguousarray(deltas)).cuda()
    om = torch.from_numpy(gen.gaussian_test_matrix(seed, D, m + p)).cuda()
    desc = pk.factor_desc(d_dev, n, T, D, m, p, q, om)
    nbytes = pk.kamera_factor_workspace_size(desc)
    ws = torch.empty(nbytes // 4 + 64, dtype=torch.float32, device="cuda")
    stride = (T + D) * m
    out = torch.full((n * stride,), -1, dtype=torch.int16, device="cuda")
    pk.kamera_factor_patches(desc, out.data_ptr(), out.data_ptr() + 2 * T * m, stride, ws.data_ptr(), nbytes,
                             pk.stream_handle())
    torch.cuda.synchronize()
    o = H.bits_to_f64(out.cpu().numpy().view(np.uint16)).reshape(n, T + D, m)
    return o[:, :T], o[:, T:]


def test_factor_largest_slab():
    """T = 8192, D = 2048 (the largest slab served), rank 64, oversample 32
    (k = 96, the largest): a deficit of exact rank 40 is reconstructed by
    U V^T to the bf16 rounding of the factors."""
    T, D = 8192, 2048
    delta = gen.low_rank_deficit(21, 0, T, D, np.linspace(9, 1, 40))[None]
    U, V = _factor(delta, m=64, p=32, q=1)
    assert_product_matches(U[0], V[0], delta[0].astype(np.float64), "largest slab")


@pytest.mark.parametrize("T,D", [(5, 3), (3, 40), (1, 64), (64, 1), (64, 4), (4, 64), (8, 8)])
def test_factor_slabs_smaller_than_k(T, D):
    """Slabs whose rank min(T, D) is below k: every dependent direction is
    dropped and the factors reproduce the slab exactly (to bf16 rounding).
    The last three are aligned (tensor-core path with tiny tiles; at D = 4 < m
    the output products take the fp32 fallback)."""
    rng = np.random.default_rng(T * 100 + D)
    delta = rng.standard_normal((2, T, D)).astype(np.float32)
    U, V = _factor(delta, m=8, p=16, q=2)
    for s in range(2):
        assert np.isfinite(U).all() and np.isfinite(V).all()
        assert_product_matches(U[s], V[s], delta[s].astype(np.float64), (T, D, s))


def test_factor_several_slabs_per_cta():
    """More slabs than resident CTAs (two per SM): each CTA takes three slabs in
    turn, so its stage and accumulator barriers carry their phases from one
    slab and product to the next.  Every slab is an exact rank-6 deficit of
    two 128-row tiles, and every one is reconstructed by U V^T to the bf16
    rounding of the factors -- a CTA whose barrier phases slipped would read a
    stale stage or accumulator and miss it."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n, T, D = 3 * 2 * sms, 256, 128
    deltas = np.stack([gen.low_rank_deficit(22, s, T, D, np.linspace(6, 1, 6)) for s in range(n)])
    U, V = _factor(deltas, m=8, p=16, q=2)
    for s in range(n):
        assert_product_matches(U[s], V[s], deltas[s].astype(np.float64), ("slab", s))
