"""Patch formation on the GPU (Kamera §2: the top-m SVD factors of the
deficit) against the oracle's exact one-sided Jacobi SVD.

The factors are defined only up to a rotation of the leading subspace, so
what is compared is the product U_m V_m^T (unique when sigma_m > sigma_{m+1}),
element by element, against the oracle's rank-m truncation P:

    |(U V^T)_tj - P_tj| <= 2^-8 sum_r |U_tr| |V_jr|  +  2^-8 max|P|.

The first term is the bf16 rounding of the two output factors (unit
roundoff 2^-9 each, so every term U_tr V_jr is off by at most (2u + u^2)
of itself).  The second covers the fp32 factors' own error: they come from
TF32 tensor-core products with fp32 accumulation -- the deficit read as
tf32 by truncation on the tensor-core path (a relative error below 2^-10
per operand; the operands the kernel writes itself are rounded, 2^-11), a
few products deep -- and a subspace iteration whose error,
(sigma_{m+1}/sigma_m)^(2q+1), is negligible with the gaps used here.  The
singular values (the column norms of V, U being orthonormal) are checked one
by one against the oracle's.  Where the spectrum has no gap the product is
not unique, and the GPU result must instead be within 2 % of the optimal
(Eckart-Young) error.
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


def elementwise_tol(U, V, P_ref):
    """The per-element bound of the module docstring."""
    return 2.0 ** -8 * (np.abs(U) @ np.abs(V).T) + 2.0 ** -8 * np.abs(P_ref).max()


def assert_product_matches(U, V, P_ref, what=""):
    err = np.abs(U @ V.T - P_ref)
    tol = elementwise_tol(U, V, P_ref)
    worst = float((err / tol).max())
    assert worst <= 1.0, (what, worst, float(err.max()), np.unravel_index(int(np.argmax(err / tol)), err.shape))


def assert_sigmas_match(V, delta, m):
    """sigma_i of the GPU product = |V[:, i]| (U orthonormal); against the
    oracle's Jacobi singular values, within the bf16 rounding of V (2^-8
    relative) plus the fp32/TF32 term of the product bound (2^-8 sigma_1)."""
    a = np.asarray(delta, np.float64)
    a = a.T if a.shape[0] < a.shape[1] else a
    sig_ref = oracle.jacobi_svd(a)[2][:m]
    sig = np.sort(np.linalg.norm(V, axis=0))[::-1][:m]
    assert np.all(np.abs(sig - sig_ref) <= 2.0 ** -8 * sig_ref + 2.0 ** -8 * sig_ref[0]), (sig[:4], sig_ref[:4])


@pytest.mark.parametrize("m", [8, 16, 32, 64])
def test_exact_low_rank_is_reconstructed(m):
    T, D, r = 300, 256, min(m, 6)
    deltas = np.stack([gen.low_rank_deficit(11, s, T, D, np.linspace(8, 2, r)) for s in range(3)])
    U, V = gpu_factor(deltas, m)
    for s in range(3):
        assert_product_matches(U[s], V[s], deltas[s], "vs the exact deficit")
        assert_product_matches(U[s], V[s], oracle_truncation(deltas[s], m), "vs the oracle truncation")
        assert_sigmas_match(V[s], deltas[s], r)


@pytest.mark.parametrize("T,D", [(300, 256), (129, 320), (1024, 512), (200, 576)])
def test_leading_subspace_matches_oracle_truncation(T, D):
    """A clear gap after the m-th singular value: the rank-m product is
    unique and the GPU must reproduce the oracle's."""
    m = 32
    spec = np.concatenate([np.linspace(10, 2, m), np.full(12, 0.05)])
    deltas = np.stack([gen.low_rank_deficit(12, s, T, D, spec, noise=1e-3) for s in range(2)])
    U, V = gpu_factor(deltas, m, p=16, q=2)
    for s in range(2):
        assert_product_matches(U[s], V[s], oracle_truncation(deltas[s], m), (T, D, s))
        assert_sigmas_match(V[s], deltas[s], m)


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
        assert_product_matches(U[s], V[s], oracle_truncation(deltas[s], m), (m, p, T, D, s))


@pytest.mark.parametrize("m,p,T,D", [(32, 32, 260, 196), (16, 48, 516, 132)])
def test_widest_single_column_tile(m, p, T, D):
    """k = m + p = 64: every tall product fills all 64 accumulator columns of
    the single column tile (the widest case of the aligned instance), with
    partial row tiles; the rank-m product still matches the oracle's."""
    spec = np.concatenate([np.linspace(9, 3, m), np.full(6, 0.02)])
    deltas = np.stack([gen.low_rank_deficit(19, s, T, D, spec, noise=1e-3) for s in range(2)])
    U, V = gpu_factor(deltas, m, p=p, q=2)
    for s in range(2):
        assert_product_matches(U[s], V[s], oracle_truncation(deltas[s], m), (m, p, T, D, s))
        assert_sigmas_match(V[s], deltas[s], m)


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
    # bf16 rounding of unit columns: each entry of U^T U is off by at most
    # 2^-8 |u_k| |u_l| = 2^-8; the fp32 columns themselves are orthonormal
    # to about 1e-6 (Cholesky QR, twice where needed)
    np.testing.assert_allclose(U[0].T @ U[0], np.eye(m), rtol=0, atol=2.0 ** -8 + 1e-4)


def test_rank_deficient_input_gives_zero_extra_columns():
    """rank(Delta) = 3 < m = 32: the extra factors contribute nothing."""
    T, D, m = 200, 128, 32
    delta = gen.low_rank_deficit(15, 0, T, D, [5.0, 3.0, 1.0])[None]
    U, V = gpu_factor(delta, m)
    assert np.isfinite(U).all() and np.isfinite(V).all()
    assert_product_matches(U[0], V[0], delta[0].astype(np.float64), "rank 3 < m")


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
    factors = H.bits_to_f64(H.to_bits(t["patch"])).reshape(n, T + D, m)
    for ch, key in ((0, "pool_k"), (1, "pool_v")):
        with_p = H.bits_to_f64(H.to_bits(t[key]))
        without = H.bits_to_f64(H.to_bits(t0[key]))
        for it in wl.items:
            pos = int(it["dst_pos"]) + np.arange(T)
            pages, slots = wl.block_table[0, pos // wl.page_size], pos % wl.page_size
            for layer in range(L):
                s_idx = (int(it["patch_id"]) * L + layer) * 2 + ch
                a, b = with_p[layer, pages, slots], without[layer, pages, slots]
                U, V = factors[s_idx, :T], factors[s_idx, T:]
                # each pool value is rounded to bf16 once: half an ulp of each side
                tol = elementwise_tol(U, V, deltas[s_idx]) + 0.5 * (H.ulp_bf16(a) + H.ulp_bf16(b))
                assert np.all(np.abs((a - b) - deltas[s_idx]) <= tol), (ch, s_idx)
