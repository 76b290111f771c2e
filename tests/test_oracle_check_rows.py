"""The row-block parity driver the full-size GPU tests use (CPU only).

``oracle.check_rows`` recomputes every row with the oracle's own per-row
function and applies the comparison rule in C, so that whole pools of the
largest workloads can be checked on all host cores.  Here it is pinned to
(a) the rule as the Python harness states it -- planted errors at and across
the tolerance edge, NaN, the exact-copy columns -- and (b) the oracle's row
function itself: a correctly rounded block passes, a block from a wrong
shift, a dropped patch or a transposed V fails.  ``oracle.check_rows_compressed``
(rows decoded from a compressed store first) is pinned to the oracle's whole
compressed reuse operator."""
import numpy as np
import pytest

import oracle
from synth import gen
from tests import harness as H

rng = np.random.default_rng(23)


def _bf16(x) -> np.ndarray:
    return gen.f32_to_bf16_bits(np.asarray(x, np.float64).astype(np.float32))


def _block(family=oracle.GQA, n=40, rank=16, sections=(0, 0, 0)):
    if family == oracle.MLA:
        m = oracle.model(oracle.MLA, 1, rope_dim=64, latent_dim=512, sections=sections)
        th = oracle.theta(1e4, 64)
    else:
        m = oracle.model(family, 1, 4, 128, sections=sections)
        th = oracle.theta(1e6, 128)
    D = oracle.row_dim(m)
    src = _bf16(rng.standard_normal((n, D)))
    u = _bf16(rng.standard_normal((n, rank)) * 0.3) if rank else None
    v = _bf16(rng.standard_normal((D, rank)) * 0.3) if rank else None
    return m, th, D, src, u, v


def _ref_rows(m, th, ch, delta, src, u, v, rotate=True):
    return np.stack([oracle.row(m, th, ch, delta, H.bits_to_f64(src[i]),
                                None if u is None else H.bits_to_f64(u[i]),
                                None if v is None else H.bits_to_f64(v), rotate=rotate) for i in range(len(src))])


@pytest.mark.parametrize("ch", [0, 1])
def test_correctly_rounded_block_passes_and_counts_match_the_harness(ch):
    m, th, D, src, u, v = _block()
    ref = _ref_rows(m, th, ch, 12345, src, u, v)
    got = _bf16(ref)
    assert oracle.check_rows(m, th, ch, 12345, src, got, u, v)[0] == 0
    # plant errors of 1..4 ulps (and a NaN) at random places: the C rule and
    # the harness rule count the same failures
    bad = got.copy()
    idx = rng.choice(got.size, 200, replace=False)
    flat = bad.reshape(-1)
    flat[idx] = (flat[idx].astype(np.int32) + rng.integers(1, 5, 200)).astype(np.uint16)
    flat[idx[0]] = 0xFFFF
    n_bad, max_err, first = oracle.check_rows(m, th, ch, 12345, src, bad, u, v)
    want = ~H.within_tol(H.bits_to_f64(bad), ref)
    assert n_bad == int(want.sum()) > 0
    assert first == int(np.flatnonzero(want.reshape(-1))[0])
    assert np.isclose(max_err, np.nanmax(np.abs(H.bits_to_f64(bad) - ref)))


def test_tolerance_edge_is_the_harness_edge():
    """Values placed just inside and just outside ulp_bf16(ref) + 1e-3 of a
    reference: the C rule and the Python rule agree element by element,
    including references that are zero or exact powers of two."""
    m, th, D, src, _, _ = _block(rank=0)
    ref = _ref_rows(m, th, 1, 0, src, None, None)  # V rows: the canonical values themselves
    assert np.array_equal(_bf16(ref), src)
    # references: powers of two, zero, and ordinary values; the device values
    # sit near ref +- (ulp + 1e-3), on the bf16 grid
    special = np.array([0.0, 1.0, -2.0, 0.5, 2.0 ** -10, 3.0, -1e-4, 7.5], np.float64)
    src2 = src.copy()
    src2[0, :special.size] = _bf16(special)
    ref2 = _ref_rows(m, th, 1, 0, src2, None, None)
    tol = H.ulp_bf16(ref2) + H.ABS_TOL
    for sgn in (1.0, -1.0):
        for k in (0.97, 1.0, 1.03, 1.2):
            got = _bf16(ref2 + sgn * k * tol)
            n_bad = oracle.check_rows(m, th, 1, 0, src2, got, rotate=False)[0]
            assert n_bad == int((~H.within_tol(H.bits_to_f64(got), ref2)).sum())


def test_exact_columns_demand_identical_bits():
    m, th, D, src, _, _ = _block(oracle.MLA, rank=0)
    ref = _ref_rows(m, th, 0, -777, src, None, None)
    got = _bf16(ref)
    assert np.array_equal(got[:, :512], src[:, :512])  # c_KV is a copy
    assert oracle.check_rows(m, th, 0, -777, src, got, n_exact=512)[0] == 0
    bad = got.copy()
    bad[3, 100] ^= np.uint16(1)  # one ulp off in a copied column: within tolerance, not exact
    assert H.within_tol(H.bits_to_f64(bad), ref).all()
    assert oracle.check_rows(m, th, 0, -777, src, bad, n_exact=512)[0] == 1
    assert oracle.check_rows(m, th, 0, -777, src, bad, n_exact=0)[0] == 0


@pytest.mark.parametrize("family", [oracle.GQA, oracle.MLA])
def test_plausible_mistakes_in_the_device_rows_are_caught(family):
    m, th, D, src, u, v = _block(family)
    good = _bf16(_ref_rows(m, th, 0, 4096, src, u, v))
    assert oracle.check_rows(m, th, 0, 4096, src, good, u, v)[0] == 0
    mistakes = {
        "shift off by one": _ref_rows(m, th, 0, 4097, src, u, v),
        "shift sign": _ref_rows(m, th, 0, -4096, src, u, v),
        "patch dropped": _ref_rows(m, th, 0, 4096, src, None, None),
        "patch before rotation": _ref_rows(oracle.model(*_fields(m, frame=oracle.PATCH_CANONICAL_FRAME)), th, 0,
                                           4096, src, u, v),
        "no rotation": _ref_rows(m, th, 0, 4096, src, u, v, rotate=False),
    }
    for what, rows in mistakes.items():
        assert oracle.check_rows(m, th, 0, 4096, src, _bf16(rows), u, v)[0] > 0, what


def test_m_rope_section_shifts_are_applied():
    m, th, D, src, u, v = _block(sections=(16, 24, 24))
    d = np.array([100, -2000, 37], np.int64)
    good = _bf16(_ref_rows(m, th, 0, d, src, u, v))
    assert oracle.check_rows(m, th, 0, d, src, good, u, v)[0] == 0
    assert oracle.check_rows(m, th, 0, np.array([100, 100, 100]), src, good, u, v)[0] > 0


def _fields(m, frame):
    return (m.family, m.num_layers, m.num_kv_heads, m.head_dim, m.rope_dim, m.latent_dim, m.pairing, frame,
            tuple(m.sections))


def test_compressed_rows_check_against_the_oracle_operator():
    """oracle.check_rows_compressed (decode, rotate, patch, compare) agrees with
    the oracle's whole compressed reuse operator: its pool image, rounded to
    bf16, passes row block by row block; a planted error, the wrong chunk or
    the wrong shift fails."""
    from synth import workloads as W

    wl = W.gqa_video(num_layers=2, n_chunks=3, T=70, rank=16, page_size=16).replace(num_kv_heads=2)
    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim, wl.latent_dim,
                     wl.pairing, wl.patch_frame)
    th = oracle.theta(wl.rope_base, wl.rope_dim)
    arrs = H.comp_arrays(wl.random_compressed())
    cs = H.oracle_store(arrs)
    err, ref_k, ref_v, wk, wv = H.oracle_reference_compressed(wl, cs)
    assert err == 0
    D, P = wl.D, wl.page_size
    for ch, ref in ((0, ref_k), (1, ref_v)):
        for it in wl.items:
            T, c, pid = int(it["n_tokens"]), int(it["chunk_id"]), int(it["patch_id"])
            pos = int(it["dst_pos"]) + np.arange(T)
            pages, slots = wl.block_table[0, pos // P], pos % P
            for layer in range(wl.num_layers):
                got = _bf16(ref[layer, pages, slots])
                u = wl.u_rows(pid, layer, ch)
                v = wl.v_rows(pid, layer, ch)
                args = (m, th, cs, c, layer, ch, 0, int(it["delta"]))
                assert oracle.check_rows_compressed(*args, got, u, v)[0] == 0
                bad = got.copy()
                bad[T // 2, D // 3] ^= np.uint16(0x0040)  # a few ulps off
                n_bad, _, first = oracle.check_rows_compressed(*args, bad, u, v)
                assert n_bad == 1 and first == (T // 2) * D + D // 3
                other = (c + 1) % len(wl.chunk_lens)
                assert oracle.check_rows_compressed(m, th, cs, other, layer, ch, 0, int(it["delta"]), got, u,
                                                    v)[0] > 0
                if ch == 0:
                    assert oracle.check_rows_compressed(m, th, cs, c, layer, ch, 0, int(it["delta"]) + 1, got, u,
                                                        v)[0] > 0
