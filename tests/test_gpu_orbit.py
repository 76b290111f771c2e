"""Orbit patch (Kamera §3 "Reorder": one patch, averaged over permutations,
serves every ordering of a cached set): the mean of deficits sampled under
several orderings, then its rank-m factors.

Mean tolerance: the n fp32 terms are added in order (error at most
(n-1) * 2^-24 * sum|x_j| to first order) and divided once (2^-24 relative)."""
import numpy as np
import pytest

import oracle
from synth import gen
from tests.test_gpu_factor import assert_product_matches, gpu_factor, oracle_truncation

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import position_invariant_kv_kamera_gb300 as pk  # noqa: E402

U32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def gpu_mean(samples: np.ndarray, pad: int = 0) -> np.ndarray:
    n = samples.shape[0]
    per = int(np.prod(samples.shape[1:]))
    stride = per + pad
    buf = np.zeros((n, stride), np.float32)
    buf[:, :per] = samples.reshape(n, per)
    d = torch.from_numpy(buf).cuda()
    out = torch.full((per,), float("nan"), dtype=torch.float32, device="cuda")
    pk.kamera_orbit_mean(d.data_ptr(), n, stride, per, out.data_ptr(), pk.stream_handle())
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64).reshape(samples.shape[1:])


@pytest.mark.parametrize("n,shape,pad", [(1, (3, 100, 64), 0), (4, (2, 256, 512), 0), (7, (5, 33), 3),
                                         (16, (1000,), 1)])
def test_orbit_mean_matches_oracle(n, shape, pad):
    rs = np.random.default_rng(n * 100 + pad)
    samples = (rs.standard_normal((n,) + shape) * 10 ** rs.uniform(-2, 2, (n,) + shape)).astype(np.float32)
    got = gpu_mean(samples, pad)
    ref = oracle.orbit_mean(samples)
    bound = (n - 1) * U32 * np.abs(samples.astype(np.float64)).sum(axis=0) / n + 2 * U32 * np.abs(ref) + 1e-30
    assert (np.abs(got - ref) <= bound).all()


def test_orbit_patch_is_the_truncation_of_the_mean_deficit():
    """Deficits under 6 orderings share a rank-8 core (singular values 10..4)
    and differ by ordering-specific rank-2 terms, which average to singular
    values near 0.25 and below; the orbit patch of rank 8 -- the shared core,
    after a 16x gap, so the product is unique -- is the rank-8 truncation of
    their mean, element by element."""
    n_ord, T, D, m = 6, 256, 256, 8
    core = gen.low_rank_deficit(41, 0, T, D, np.linspace(10, 4, 8))
    samples = np.stack([core + gen.low_rank_deficit(42, j, T, D, [1.5, 0.5]) for j in range(n_ord)])
    mean = gpu_mean(samples).astype(np.float32)
    U, V = gpu_factor(mean[None], m, p=16, q=2)
    P_ref = oracle_truncation(oracle.orbit_mean(samples), m)
    assert_product_matches(U[0], V[0], P_ref, "orbit patch")
