"""The comparison rule the GPU parity tests apply (CPU only): planted errors
in a synthetic "device" pool must be reported, a correctly rounded pool must
pass.  Without this, a mistake in the rule could make every GPU parity test
pass vacuously."""
import numpy as np

from synth import gen
from tests import harness as H

rng = np.random.default_rng(17)


def _case():
    """A pool of 3 layers x 4 pages x 8 slots x 64 features: half the rows
    written with oracle values, the rest holding the input bits."""
    shape = (3, 4, 8, 64)
    in_bits = gen.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    wrote = rng.random(shape[:-1]) < 0.5
    ref = H.bits_to_f64(in_bits).copy()
    ref[wrote] = rng.standard_normal((int(wrote.sum()), 64)) * 3.0
    ref[wrote, :4] = 0.0                     # values at zero: the absolute term applies
    gpu = in_bits.copy()
    gpu[wrote] = gen.f32_to_bf16_bits(ref[wrote].astype(np.float32))  # round to nearest even
    return in_bits, ref, wrote, gpu


def test_correctly_rounded_pool_passes():
    in_bits, ref, wrote, gpu = _case()
    rep = H.compare_pool(gpu, in_bits, ref, wrote)
    assert rep["untouched_bit_exact"] and rep["within_tol"] and rep["n_bad"] == 0
    assert rep["rows_written"] == int(wrote.sum())


def test_truncated_pool_passes_but_two_ulp_error_fails():
    in_bits, ref, wrote, gpu = _case()
    # truncation toward zero stays within one ulp of the exact value
    trunc = in_bits.copy()
    trunc[wrote] = (ref[wrote].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert H.compare_pool(trunc, in_bits, ref, wrote)["within_tol"]
    # one element three ulps off (above the absolute term) is caught
    idx = tuple(np.argwhere(wrote)[0])
    row = H.bits_to_f64(gpu[idx])
    j = int(np.argmax(np.abs(row)))
    bad = gpu.copy()
    bad[idx + (j,)] = np.uint16(int(bad[idx + (j,)]) + 3)
    rep = H.compare_pool(bad, in_bits, ref, wrote)
    assert not rep["within_tol"] and rep["n_bad"] == 1


def test_nan_and_unwritten_sentinel_in_a_written_row_fail():
    in_bits, ref, wrote, gpu = _case()
    idx = tuple(np.argwhere(wrote)[1])
    bad = gpu.copy()
    bad[idx + (5,)] = np.uint16(0xFFFF)      # the sentinel: a bf16 NaN
    assert not H.compare_pool(bad, in_bits, ref, wrote)["within_tol"]


def test_a_changed_untouched_slot_fails():
    in_bits, ref, wrote, gpu = _case()
    idx = tuple(np.argwhere(~wrote)[0])
    bad = gpu.copy()
    bad[idx + (0,)] ^= np.uint16(1)          # one bit of one untouched slot
    rep = H.compare_pool(bad, in_bits, ref, wrote)
    assert not rep["untouched_bit_exact"] and rep["within_tol"]


def test_exact_columns_demand_identical_bits():
    in_bits, ref, wrote, gpu = _case()
    ref2 = ref.copy()
    ref2[wrote, :32] = H.bits_to_f64(gpu[wrote, :32])   # the copied columns: exact bf16 values
    assert H.compare_pool(gpu, in_bits, ref2, wrote, exact_cols=slice(0, 32))["exact_cols_bit_exact"]
    idx = tuple(np.argwhere(wrote)[2])
    bad = gpu.copy()
    bad[idx + (7,)] ^= np.uint16(1)          # one ulp in a copied column: within tolerance, not exact
    rep = H.compare_pool(bad, in_bits, ref2, wrote, exact_cols=slice(0, 32))
    assert rep["within_tol"] and not rep["exact_cols_bit_exact"]


def test_ulp_is_the_bf16_spacing():
    x = np.array([1.0, 1.5, 2.0, -3.0, 0.75, 1e-3, 0.0])
    np.testing.assert_array_equal(H.ulp_bf16(x)[:6], [2 ** -7, 2 ** -7, 2 ** -6, 2 ** -6, 2 ** -8, 2 ** -17])
    assert H.ulp_bf16(x)[6] == 2.0 ** -133
