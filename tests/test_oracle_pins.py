"""Pins of the fp64 oracle to facts fixed by the Kamera page and by mathematics,
not by the oracle itself (CPU only).

Kamera §2 "Relocation R(delta)": keys re-rotated by the RoPE phase shift of
the new position, an exact algebraic operation.  The pins below use
independent formulations: complex exponentials, a matrix exponential of the
rotation generator, library SVD, brute-force index maps.
"""
import json
import os

import numpy as np
import pytest
import scipy.linalg

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _theta_np(base, d):
    # RoPE frequency ladder written independently of the oracle
    return np.exp(-np.log(base) * np.arange(0, d, 2) / d)


def rope_complex(x, pos, theta, pairing=oracle.ROTATE_HALF):
    """RoPE of a d-vector at integer position pos as complex multiplication
    z_i * exp(i * pos * theta_i)."""
    d = x.shape[0]
    h = d // 2
    if pairing == oracle.ROTATE_HALF:
        z = x[:h] + 1j * x[h:]
    else:
        z = x[0::2] + 1j * x[1::2]
    z = z * np.exp(1j * pos * theta)
    out = np.empty_like(x)
    if pairing == oracle.ROTATE_HALF:
        out[:h], out[h:] = z.real, z.imag
    else:
        out[0::2], out[1::2] = z.real, z.imag
    return out


def test_theta_matches_independent_ladder(oracle_lib):
    for base, d in [(1e4, 64), (1e6, 128), (5e5, 128), (1e4, 256)]:
        np.testing.assert_allclose(oracle.theta(base, d), _theta_np(base, d), rtol=1e-14, atol=0)
    assert oracle.theta(1e4, 64)[0] == 1.0


@pytest.mark.parametrize("pairing", [oracle.ROTATE_HALF, oracle.INTERLEAVED])
@pytest.mark.parametrize("d,base", [(64, 1e4), (128, 1e6)])
def test_rerotation_equals_rope_at_shifted_position(oracle_lib, pairing, d, base):
    """rope(x, p) re-rotated by delta equals rope(x, p + delta)."""
    th = _theta_np(base, d)
    for p, delta in [(0, 1000), (17, -5), (4096, 32768), (100000, -99999), (3, 0)]:
        x = rng.standard_normal(d)
        got = oracle.rotate_region(rope_complex(x, p, th, pairing), th, delta, pairing)
        want = rope_complex(x, p + delta, th, pairing)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-9)


@pytest.mark.parametrize("pairing", [oracle.ROTATE_HALF, oracle.INTERLEAVED])
def test_group_law_and_inverse(oracle_lib, pairing):
    th = oracle.theta(1e6, 128)
    for d1, d2 in [(1000, 2345), (-32768, 32768), (7, -9), (150000, 57000)]:
        x = rng.standard_normal(128)
        two = oracle.rotate_region(oracle.rotate_region(x, th, d1, pairing), th, d2, pairing)
        one = oracle.rotate_region(x, th, d1 + d2, pairing)
        np.testing.assert_allclose(two, one, rtol=0, atol=1e-9)
        back = oracle.rotate_region(oracle.rotate_region(x, th, d1, pairing), th, -d1, pairing)
        np.testing.assert_allclose(back, x, rtol=0, atol=1e-10)


def test_delta_zero_is_identity(oracle_lib):
    th = oracle.theta(1e4, 64)
    x = rng.standard_normal(64)
    np.testing.assert_array_equal(oracle.rotate_region(x, th, 0), x)


@pytest.mark.parametrize("pairing", [oracle.ROTATE_HALF, oracle.INTERLEAVED])
def test_rotation_is_matrix_exponential_of_generator(oracle_lib, pairing):
    """R(delta) = expm(delta * A), A block-skew with rates theta_i on each pair."""
    d = 64
    th = oracle.theta(1e4, d)
    A = np.zeros((d, d))
    for i in range(d // 2):
        a, b = (i, i + d // 2) if pairing == oracle.ROTATE_HALF else (2 * i, 2 * i + 1)
        A[b, a], A[a, b] = th[i], -th[i]
    for delta in [1, 7, -3, 25]:
        R = scipy.linalg.expm(delta * A)
        x = rng.standard_normal(d)
        np.testing.assert_allclose(oracle.rotate_region(x, th, delta, pairing), R @ x, rtol=0, atol=1e-11)


def test_rotation_preserves_pair_norms(oracle_lib):
    th = oracle.theta(5e5, 128)
    x = rng.standard_normal(128)
    y = oracle.rotate_region(x, th, -8192)
    np.testing.assert_allclose(np.hypot(y[:64], y[64:]), np.hypot(x[:64], x[64:]), rtol=1e-13)


def test_row_rotates_every_head_and_only_keys(oracle_lib):
    m = oracle.model(oracle.GQA, 1, num_kv_heads=4, head_dim=128)
    th = oracle.theta(1e6, 128)
    x = rng.standard_normal(512)
    k = oracle.rotate_row(m, th, 0, 321, x)
    for h in range(4):
        np.testing.assert_allclose(k[h * 128:(h + 1) * 128], rope_complex(x[h * 128:(h + 1) * 128], 321, th),
                                   atol=1e-11)
    np.testing.assert_array_equal(oracle.rotate_row(m, th, 1, 321, x), x)  # V: no position


def test_partial_rotary_leaves_tail_untouched(oracle_lib):
    m = oracle.model(oracle.GQA, 1, num_kv_heads=2, head_dim=128, rope_dim=64)
    th = oracle.theta(1e4, 64)
    x = rng.standard_normal(256)
    k = oracle.rotate_row(m, th, 0, 99, x)
    for h in range(2):
        np.testing.assert_allclose(k[h * 128:h * 128 + 64], rope_complex(x[h * 128:h * 128 + 64], 99, th), atol=1e-11)
        np.testing.assert_array_equal(k[h * 128 + 64:(h + 1) * 128], x[h * 128 + 64:(h + 1) * 128])


def test_mla_rotates_only_k_rope(oracle_lib):
    """Kamera §2, MLA: only the decoupled 64-dim k_rope is relocated; c_KV is
    reused byte for byte."""
    m = oracle.model(oracle.MLA, 1, rope_dim=64, latent_dim=512)
    th = oracle.theta(1e4, 64)
    x = rng.standard_normal(576)
    y = oracle.rotate_row(m, th, 0, -4444, x)
    np.testing.assert_array_equal(y[:512], x[:512])
    np.testing.assert_allclose(y[512:], rope_complex(x[512:], -4444, th), atol=1e-11)


def test_patch_is_low_rank_product(oracle_lib):
    """Kamera §2, patch application: out = R src + U V^T (checked with a library matmul)."""
    m = oracle.model(oracle.GQA, 1, num_kv_heads=2, head_dim=64)
    th = oracle.theta(1e4, 64)
    D, r, T = 128, 16, 9
    src = rng.standard_normal((T, D))
    U = rng.standard_normal((T, r))
    V = rng.standard_normal((D, r))
    P = U @ V.T
    for t in range(T):
        for ch in (0, 1):
            got = oracle.row(m, th, ch, 0, src[t], U[t], V)
            np.testing.assert_allclose(got, src[t] + P[t], atol=1e-12)
            got = oracle.row(m, th, ch, 77, src[t], U[t], V)
            want = oracle.rotate_row(m, th, ch, 77, src[t]) + P[t]
            np.testing.assert_allclose(got, want, atol=1e-12)


def test_one_hot_patch_changes_one_element(oracle_lib):
    m = oracle.model(oracle.GQA, 1, num_kv_heads=1, head_dim=64)
    th = oracle.theta(1e4, 64)
    src = rng.standard_normal(64)
    u = np.zeros(8)
    u[3] = 0.5
    V = np.zeros((64, 8))
    V[41, 3] = -2.0
    base = oracle.row(m, th, 0, 5, src)
    got = oracle.row(m, th, 0, 5, src, u, V)
    diff = got - base
    assert np.count_nonzero(diff) == 1 and diff[41] == -1.0


def test_canonical_frame_equals_rotated_factor_patch(oracle_lib):
    """R(d)(k + U V^T) = R(d) k + U (R(d) V)^T: the canonical-frame reading is
    again rank m, with V's feature axis rotated."""
    mc = oracle.model(oracle.GQA, 1, num_kv_heads=2, head_dim=64, patch_frame=oracle.PATCH_CANONICAL_FRAME)
    ma = oracle.model(oracle.GQA, 1, num_kv_heads=2, head_dim=64)
    th = oracle.theta(1e4, 64)
    src = rng.standard_normal(128)
    u = rng.standard_normal(8)
    V = rng.standard_normal((128, 8))
    RV = np.stack([oracle.rotate_row(ma, th, 0, 1234, V[:, j]) for j in range(8)], axis=1)
    got = oracle.row(mc, th, 0, 1234, src, u, V)
    want = oracle.row(ma, th, 0, 1234, src, u, RV)
    np.testing.assert_allclose(got, want, atol=1e-11)


def test_slot_mapping_brute_force(oracle_lib):
    P, n_seqs, mp, num_pages = 16, 3, 5, 20
    bt = rng.permutation(num_pages)[: n_seqs * mp].reshape(n_seqs, mp).astype(np.int32)
    bt[1, 4] = 25  # out of range page id
    bt[2, 0] = -1
    for seq in range(n_seqs):
        for pos in range(-2, mp * P + 3):
            want = -1
            if 0 <= pos < mp * P:
                page = int(bt[seq, pos // P])
                if 0 <= page < num_pages:
                    want = page * P + pos % P
            assert oracle.slot(bt, mp, num_pages, P, seq, pos) == want


def test_patch_byte_accounting_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "patch_bytes.json")))
    T, D = g["T"], g["D"]
    for case in g["cases"]:
        frac = (T + D) * case["rank"] / (T * D)
        assert abs(frac - case["approx_fraction"]) <= case["abs_tol"]


def _svd_case(rows, cols, r, seed):
    g = np.random.default_rng(seed)
    A = g.standard_normal((rows, r))
    B = g.standard_normal((cols, r))
    return A @ B.T


@pytest.mark.parametrize("rows,cols,r,m", [(40, 12, 3, 3), (40, 12, 3, 5), (64, 16, 8, 8), (30, 30, 1, 4)])
def test_jacobi_svd_reconstructs_exact_rank(oracle_lib, rows, cols, r, m):
    """A deficit of exact rank r, factored and truncated to m >= r, is
    reconstructed exactly (Kamera §2: top-m SVD factors form the patch)."""
    delta = _svd_case(rows, cols, r, rows * cols + r)
    us, v, sig = oracle.jacobi_svd(delta)
    Um, Vm = us[:, :m], v[:, :m]
    np.testing.assert_allclose(Um @ Vm.T, delta, atol=1e-10 * np.abs(delta).max())
    np.testing.assert_allclose(sig, np.linalg.svd(delta, compute_uv=False), atol=1e-10 * sig[0])


def test_jacobi_svd_truncation_residual_is_eckart_young(oracle_lib):
    g = np.random.default_rng(5)
    a = g.standard_normal((50, 20))
    us, v, sig = oracle.jacobi_svd(a)
    for m in (1, 4, 10, 19):
        resid = np.linalg.norm(a - us[:, :m] @ v[:, :m].T)
        np.testing.assert_allclose(resid, np.sqrt((sig[m:] ** 2).sum()), rtol=1e-10)
    np.testing.assert_allclose(v.T @ v, np.eye(20), atol=1e-12)


def mrope_complex(x, pos3, theta, sections, pairing=oracle.ROTATE_HALF):
    """M-RoPE written as complex multiplication: pair i of section s turns by
    pos3[s] * theta_i (sections = consecutive runs of pairs)."""
    h = x.shape[0] // 2
    sec_of = np.repeat(np.arange(3), sections)
    phase = np.asarray(pos3, np.float64)[sec_of] * theta
    if pairing == oracle.ROTATE_HALF:
        z = (x[:h] + 1j * x[h:]) * np.exp(1j * phase)
        return np.concatenate([z.real, z.imag])
    z = (x[0::2] + 1j * x[1::2]) * np.exp(1j * phase)
    out = np.empty_like(x)
    out[0::2], out[1::2] = z.real, z.imag
    return out


@pytest.mark.parametrize("pairing", [oracle.ROTATE_HALF, oracle.INTERLEAVED])
def test_mrope_sections_shift_each_position_component(oracle_lib, pairing):
    """Multimodal RoPE (temporal / height / width sections, e.g. 16/24/24 pairs
    of a 128-dim head): re-rotating by (dt, dh, dw) moves each component."""
    th = _theta_np(1e6, 128)
    sec = (16, 24, 24)
    for p3, d3 in [((5, 7, 9), (1000, -3, 0)), ((0, 0, 0), (32768, 17, -17)), ((100, 2, 3), (0, 0, 0))]:
        x = rng.standard_normal(128)
        got = oracle.rotate_region_sections(mrope_complex(x, p3, th, sec, pairing), th, d3, sec, pairing)
        want = mrope_complex(x, np.add(p3, d3), th, sec, pairing)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-9)


def test_mrope_equal_shifts_is_plain_rope_and_group_law(oracle_lib):
    th = oracle.theta(1e6, 128)
    sec = (16, 24, 24)
    x = rng.standard_normal(128)
    np.testing.assert_array_equal(oracle.rotate_region_sections(x, th, (77, 77, 77), sec),
                                  oracle.rotate_region(x, th, 77))
    a = oracle.rotate_region_sections(oracle.rotate_region_sections(x, th, (5, -9, 100), sec), th, (-2, 9, 1), sec)
    np.testing.assert_allclose(a, oracle.rotate_region_sections(x, th, (3, 0, 101), sec), atol=1e-11)
    # no sections: every pair takes the first shift
    np.testing.assert_array_equal(oracle.rotate_region_sections(x, th, (5, 6, 7), (0, 0, 0)),
                                  oracle.rotate_region(x, th, 5))


def test_orbit_mean_is_the_library_mean(oracle_lib):
    """Kamera §3 reorder: the orbit deficit is the mean over sampled orderings."""
    d = rng.standard_normal((5, 7, 33)).astype(np.float32)
    np.testing.assert_allclose(oracle.orbit_mean(d), d.astype(np.float64).mean(axis=0), rtol=0, atol=1e-15)
    one = rng.standard_normal((1, 10)).astype(np.float32)
    np.testing.assert_array_equal(oracle.orbit_mean(one), one[0].astype(np.float64))
