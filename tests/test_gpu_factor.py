"""Patch formation on the GPU (Kamera §2: the top-m SVD factors of the
deficit) against the oracle's exact one-sided Jacobi SVD.

The factors are defined only up to a rotation of the leading subspace, so
what is compared is the product U_m V_m^T (unique when sigma_m > sigma_{m+1}).
Tolerances: the factors are rounded to bf16 (8 significant bits), so the
product carries a relative error of about 2^-8 -- 1e-2 of its Frobenius norm
is allowed; where the spectrum has no gap the GPU result must be within 2 %
of the optimal (Eckart-Young) error.
"""
import numpy as np
import pytest

import oracle
from synth import gen
from tests import harness as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import position_invariant_kv_kamera_gb300 as pk  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def gpu_factor(deltas: np.ndarray, m: int, p: int = 16, q: int = 2, seed: int = 5):
    """deltas [n][T][D] fp32 -> (U [n][T][m], V [n][D][m]) as fp64 from the bf16 outputs."""
    n, T, D = deltas.shape
    k = m + p
    d_dev = torch.from_numpy(np.ascontiguousarray(deltas)).cuda()
    om = torch.from_numpy(gen.gaussian_test_matrix(seed, D, k)).cuda()
    desc = pk.factor_desc(d_dev, n, T, D, m, p, q, om)
    ws_bytes = pk.kamera_factor_workspace_size(desc)
    ws = torch.empty(ws_bytes // 4 + 64, dtype=torch.float32, device="cuda")
    stride = (T + D) * m  # the patch-store layout: U then V per slab
    out = torch.full((n * stride,), -1, dtype=torch.int16, device="cuda")
    pk.kamera_factor_patches(desc, out.data_ptr(), out.data_ptr() + 2 * T * m, stride, ws.data_ptr(), ws_bytes,
                             pk.stream_handle())
    torch.cuda.synchronize()
    o = H.bits_to_f64(out.cpu().numpy().view(np.uint16)).reshape(n, T + D, m)
    return o[:, :T], o[:, T:]


def oracle_truncation(delta: np.ndarray, m: int) -> np.ndarray:
    """Rank-m truncation of delta from the oracle's Jacobi SVD (fp64)."""
    a = np.asarray(delta, np.float64)
    tr = a.shape[0] < a.shape[1]
    if tr:
        a = a.T
    us, v, sig = oracle.jacobi_svd(a)
    p = us[:, :m] @ v[:, :m].T
    return p.T if tr else p


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


@pytest.mark.parametrize("m", [8, 16, 32, 64])
def test_exact_low_rank_is_reconstructed(m):
    T, D, r = 300, 256, min(m, 6)
    deltas = np.stack([gen.low_rank_deficit(11, s, T, D, np.linspace(8, 2, r)) for s in range(3)])
    U, V = gpu_factor(deltas, m)
    for s in range(3):
        P = U[s] @ V[s].T
        assert rel(P, deltas[s]) < 1e-2
        assert rel(P, oracle_truncation(deltas[s], m)) < 1e-2


@pytest.mark.parametrize("T,D", [(300, 256), (129, 320), (1024, 512), (200, 576)])
def test_leading_subspace_matches_oracle_truncation(T, D):
    """A clear gap after the m-th singular value: the rank-m product is
    unique and the GPU must reproduce the oracle's."""
    m = 32
    spec = np.concatenate([np.linspace(10, 2, m), np.full(12, 0.05)])
    deltas = np.stack([gen.low_rank_deficit(12, s, T, D, spec, noise=1e-3) for s in range(2)])
    U, V = gpu_factor(deltas, m, p=16, q=2)
    for s in range(2):
        P_ref = oracle_truncation(deltas[s], m)
        assert rel(U[s] @ V[s].T, P_ref) < 1e-2


@pytest.mark.parametrize("m,p,T,D", [(8, 12, 260, 196), (16, 20, 132, 516), (32, 4, 388, 100), (8, 40, 64, 64)])
def test_oversampling_that_leaves_partial_tiles(m, p, T, D):
    """k = m + p not a multiple of 8 or 16 (k = 20, 36, 36, 48) and T, D off
    the 128-row tile: the last output tile and the last column tile are
    partial; the rank-m product still matches the oracle's truncation."""
    spec = np.concatenate([np.linspace(9, 3, m), np.full(6, 0.02)])
    deltas = np.stack([gen.low_rank_deficit(17, s, T, D, spec, noise=1e-3) for s in range(2)])
    U, V = gpu_factor(deltas, m, p=p, q=2)
    for s in range(2):
        assert np.isfinite(U[s]).all() and np.isfinite(V[s]).all()
        assert rel(U[s] @ V[s].T, oracle_truncation(deltas[s], m)) < 1e-2


def test_near_optimal_without_a_gap():
    """Slowly decaying spectrum: the error is within 2 % of Eckart-Young."""
    T, D, m = 256, 192, 16
    spec = 10.0 * 0.9 ** np.arange(80)
    delta = gen.low_rank_deficit(13, 0, T, D, spec)[None]
    U, V = gpu_factor(delta, m, p=24, q=3)
    P_opt = oracle_truncation(delta[0], m)
    err_gpu = np.linalg.norm(delta[0] - U[0] @ V[0].T)
    err_opt = np.linalg.norm(delta[0] - P_opt)
    assert err_gpu <= 1.02 * err_opt + 1e-2 * np.linalg.norm(P_opt)


def test_u_has_orthonormal_columns():
    T, D, m = 300, 256, 16
    delta = gen.low_rank_deficit(14, 0, T, D, np.linspace(9, 1, 24))[None]
    U, V = gpu_factor(delta, m)
    np.testing.assert_allclose(U[0].T @ U[0], np.eye(m), atol=2e-2)


def test_rank_deficient_input_gives_zero_extra_columns():
    """rank(Delta) = 3 < m = 32: the extra factors contribute nothing."""
    T, D, m = 200, 128, 32
    delta = gen.low_rank_deficit(15, 0, T, D, [5.0, 3.0, 1.0])[None]
    U, V = gpu_factor(delta, m)
    P = U[0] @ V[0].T
    assert rel(P, delta[0]) < 1e-2
    assert np.isfinite(U).all() and np.isfinite(V).all()


def test_zero_deficit_gives_zero_factors():
    U, V = gpu_factor(np.zeros((2, 100, 64), np.float32), 8)
    assert np.all(U @ np.swapaxes(V, 1, 2) == 0)


def test_formed_patch_feeds_the_reuse_operator():
    """Factors written straight into a patch store are what kamera_reuse_batched
    applies: with an exact low-rank deficit, reuse-with-patch minus
    reuse-without-patch reproduces the deficit (a generator input), within
    the bf16 rounding of the two outputs."""
    from synth import workloads as W

    wl = W.gqa_video(num_layers=2, n_chunks=2, T=256, rank=16, page_size=64)
    T, D, m, L = 256, wl.D, 16, wl.num_layers
    n = len(wl.patch_lens) * L * 2  # slab order = patch-store order: (patch, layer, channel)
    spec = 100.0 * np.linspace(4, 1, 6)
    deltas = np.stack([gen.low_rank_deficit(16, s, T, D, spec) for s in range(n)])
    t = H.device_inputs(wl, torch)
    d_dev = torch.from_numpy(deltas).cuda()
    om = torch.from_numpy(gen.gaussian_test_matrix(6, D, m + 16)).cuda()
    desc = pk.factor_desc(d_dev, n, T, D, m, 16, 1, om)
    nbytes = pk.kamera_factor_workspace_size(desc)
    ws = torch.empty(nbytes // 4 + 64, dtype=torch.float32, device="cuda")
    base = t["patch"].data_ptr()
    pk.kamera_factor_patches(desc, base, base + 2 * T * m, (T + D) * m, ws.data_ptr(), nbytes, pk.stream_handle())
    H.call(wl, t)
    t0 = H.device_inputs(wl.replace(rank=0, patch_lens=[]), torch)
    H.call(wl.replace(rank=0, patch_lens=[]), t0)
    torch.cuda.synchronize()
    assert int(t["err"].item()) == 0
    for ch, key in ((0, "pool_k"), (1, "pool_v")):
        with_p = H.bits_to_f64(H.to_bits(t[key]))
        without = H.bits_to_f64(H.to_bits(t0[key]))
        for it in wl.items:
            pos = int(it["dst_pos"]) + np.arange(T)
            pages, slots = wl.block_table[0, pos // wl.page_size], pos % wl.page_size
            for layer in range(L):
                s_idx = (int(it["patch_id"]) * L + layer) * 2 + ch
                diff = with_p[layer, pages, slots] - without[layer, pages, slots]
                assert rel(diff, deltas[s_idx]) < 2e-2
