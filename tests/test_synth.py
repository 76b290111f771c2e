"""The seeded input generator and the workload recipe (CPU only).

The generator is pinned to the published splitmix64 outputs and to the
moments of the Irwin-Hall sum; the bf16 conversion to round-to-nearest-even
at exact ties; the workloads to the recipe they stand for (N(0,1) rows with
about 1 % outlier channels x8, N(0, 0.02) patch factors, shifts uniform in
[-32768, 32768], a shuffled page table); and the byte and flop accounting
that the benchmark's roofline divides by to closed forms per unit of work."""
import numpy as np
import pytest

from synth import gen
from synth import workloads as W


def test_splitmix64_published_outputs():
    # the first five outputs of the reference splitmix64 generator (Steele, Lea
    # & Flood 2014; Vigna's splitmix64.c) seeded with 1234567
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    assert [int(x) for x in gen.hash64(1234567, np.arange(5, dtype=np.uint64))] == want


def test_bf16_rounding_is_nearest_even_at_ties():
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -20, 3.0, 2 ** -130],
                 np.float32)
    got = (gen.f32_to_bf16_bits(x).astype(np.uint32) << 16).view(np.float32)
    want = np.array([1.0, 1 + 2 ** -6, -1.0, 1 + 2 ** -7, 3.0, 2 ** -130], np.float32)
    np.testing.assert_array_equal(got, want)
    # away from ties: the nearest bf16 value, within half a bf16 ulp
    rng = np.random.default_rng(4)
    v = (rng.standard_normal(20000) * 10).astype(np.float32)
    b = (gen.f32_to_bf16_bits(v).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.abs(v.astype(np.float64)))) - 7)
    assert np.all(np.abs(b - v) <= ulp / 2)


def test_irwin_hall_normals_have_unit_moments_and_bounded_tails():
    x = gen.normal_f32(gen.stream_id(9, 1), np.arange(1 << 20, dtype=np.uint64))
    assert abs(float(x.mean())) < 0.005
    assert abs(float(x.std()) - 1.0) < 0.005
    assert float(np.abs(x).max()) <= 131070 / gen.IH_SD + 1e-3   # the sum's range ends at about 3.46 sd
    # the kurtosis of the sum of four uniforms: 3 - 6/(5*4) = 2.7
    k = float(np.mean(x.astype(np.float64) ** 4) / np.mean(x.astype(np.float64) ** 2) ** 2)
    assert abs(k - 2.7) < 0.02


def test_headline_rows_have_one_percent_outlier_channels_at_eight_sigma():
    wl = W.gqa_video()
    stds = []
    for layer in range(wl.num_layers):
        for ch in range(2):
            rows = wl.store_rows(3, layer, ch, 0, 128)
            v = (rows.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            s = v.std(axis=0)
            stds.append(s)
    s = np.concatenate(stds)
    outlier = s > 3.0
    frac = outlier.mean()
    assert 0.006 < frac < 0.014, frac                   # about 1 % of the channels
    assert abs(np.median(s[outlier]) - 8.0) < 0.8       # scaled x8
    assert abs(np.median(s[~outlier]) - 1.0) < 0.1      # the rest N(0, 1)


def test_headline_patch_factors_deltas_and_page_table():
    wl = W.gqa_video()
    u = (wl.u_rows(0, 0, 0).astype(np.uint32) << 16).view(np.float32)
    v = (wl.v_rows(5, 7, 1).astype(np.uint32) << 16).view(np.float32)
    assert abs(float(u.std()) - 0.02) < 0.001 and abs(float(v.std()) - 0.02) < 0.001
    d = wl.items["delta"]
    assert d.min() >= -32768 and d.max() <= 32768 and len(np.unique(d)) == len(d)
    bt = wl.block_table
    assert sorted(bt.ravel().tolist()) == list(range(wl.num_pages))
    assert not np.array_equal(bt.ravel(), np.arange(wl.num_pages))  # shuffled


def _per_unit_bytes(name, wl):
    """Closed forms per (item, layer): bf16 K/V rows read and written once,
    patch factors read once."""
    T = wl.items["n_tokens"].astype(np.int64)
    L, D, m = wl.num_layers, wl.D, wl.rank
    has_patch = (wl.items["patch_id"] >= 0) & (m > 0)
    if name == "sliding_window":
        return int((L * T * D * 2 * 2).sum())                       # K only, in place
    if wl.family == W.MLA:
        return int((L * (T * D * 2 * 2 + has_patch * (T + D) * m * 2)).sum())
    return int((L * 2 * (T * D * 2 * 2 + has_patch * (T + D) * m * 2)).sum())


@pytest.mark.parametrize("name,bytes_,flops", [
    ("tiny_mha", 540_672, 2 * 8 * 256 * 256 * 2),
    ("gqa_video", 1_967_128_576, 2 * 32 * 16 * 1024 * 512 * 2 * 28),
    ("mla_lite", 1_037_352_960, 2 * 16 * 8 * 2048 * 576 * 27),
    ("sliding_window", 7_516_192_768, 0),
    ("long_video", 57_399_050_240, 2 * 64 * 160 * 1296 * 1024 * 2 * 32),
])
def test_algorithmic_bytes_and_patch_flops_per_workload(name, bytes_, flops):
    wl = W.WORKLOADS[name]()
    assert wl.algorithmic_bytes() == bytes_ == _per_unit_bytes(name, wl)
    assert wl.patch_flops() == flops


def test_compressed_bytes_closed_form():
    wl = W.gqa_video()
    T, L, D, H, m = 1024, 28, 512, 4, 32
    per_item = L * T * (D + 3 * D // 8 + 4 * H) + L * 2 * T * D * 2 + L * 2 * (T + D) * m * 2
    assert wl.compressed_bytes() == 16 * per_item == 1_357_905_920
