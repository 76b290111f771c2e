"""Host-side figures of the benchmark line (CPU only): the algorithmic flops
of patch formation, and the DRAM traffic read from a profile summary, which
the line reports only while the profiled kernel sources are unchanged."""
import pytest

import bench


def test_patch_formation_flops_per_slab_and_launch():
    # T = 1024, D = 512, k = m + p = 48, m = 32, q = 2:
    # products 2TDk(2 + 2q) + 2Dk^2 + 2(T + D)km, one QR per panel 2k^2(T + q(T + D))
    per_slab = (2 * 1024 * 512 * 48 * 6 + 2 * 512 * 48 * 48 + 2 * 1536 * 48 * 32
                + 2 * 48 * 48 * (1024 + 2 * 1536))
    assert per_slab == 327_942_144
    assert bench.factor_flops(1024, 512, 48, 32, 2) == per_slab
    assert 896 * per_slab == pytest.approx(2.938e11, rel=1e-3)


def test_traffic_comes_from_a_capture_of_the_current_sources_only(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for f in bench.KERNEL_SOURCES:
        (tmp_path / f).parent.mkdir(parents=True, exist_ok=True)
        (tmp_path / f).write_text("// kernel source v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.kernel_hash()
    (prof / "reuse_kernel_full.md").write_text(f"kernel_sources_sha256_16: {h}\ndram_bytes_per_launch: 1234\n")
    (prof / "reuse_kernel_reduced.md").write_text(
        f"kernel_sources_sha256_16: {h}\ndram_bytes_per_launch_reduced: 100\ntraffic_scale_to_full: 20.0\n")
    assert bench.profile_traffic("full") == 1234
    assert bench.profile_traffic("reduced") == 2000
    assert bench.profile_traffic("missing") is None
    # once a kernel source changes, the capture no longer describes the kernel
    (tmp_path / bench.KERNEL_SOURCES[0]).write_text("// kernel source v2\n")
    assert bench.profile_traffic("full") is None and bench.profile_traffic("reduced") is None


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
