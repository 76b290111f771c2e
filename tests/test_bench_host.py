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


def test_patch_formation_bytes_are_six_delta_reads_plus_the_factors():
    # q = 2: Y, (Z, Y) twice, B -> 6 fp32 reads of each 1024 x 512 slab; U_m, V_m bf16 once
    per_slab = 6 * 1024 * 512 * 4 + (1024 + 512) * 32 * 2
    assert bench.factor_bytes(896, 1024, 512, 32, 2) == 896 * per_slab
    assert 896 * 6 * 1024 * 512 * 4 == pytest.approx(11.27e9, rel=1e-3)


def test_host_cores_and_the_oracle_sample_shapes():
    assert bench.host_cores() >= 1
    for name in ("gqa_video", "mla_lite", "long_video", "sliding_window"):
        full = bench.W.WORKLOADS[name]()
        wl = bench.oracle_sample_workload(name, 1, 128)
        # the same layers, row width, rank and page size as the workload; one chunk, truncated
        assert (wl.num_layers, wl.D, wl.rank, wl.page_size, wl.mode) == (
            full.num_layers, full.D, full.rank, full.page_size, full.mode)
        assert len(wl.items) == 1 and int(wl.items["n_tokens"][0]) == 128


def test_configs_cover_the_other_four_workloads():
    assert sorted(bench.CONFIG_ORDER + ["long_video"]) == sorted(bench.W.WORKLOADS)


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
