"""The oracle's pins catch plausible mistakes (CPU only).

Each mutant plants one mistake -- a flipped sign, a swapped or shifted index,
a dropped term, a transposed operand, an off-by-one -- into a copy of the
oracle's C source, builds it, and runs the independent checks below (complex
RoPE, M-RoPE, library matmul, brute-force page map, the vectorised whole-batch
formulation, library SVD, library mean, Max's quantiser table, the int8 error
bound, scipy's Hadamard matrix, the nearest-centroid rule, the error bits of
items that disagree with the stores).  Every mutant must fail at least one.
"""

import json
import os

import numpy as np
import pytest
from scipy import linalg

import oracle
from synth import gen
from synth import workloads as W
from tests.test_oracle_compressed import _independent_reuse_compressed, _pack, _unpack, check_store_encoding
from tests.test_oracle_operator import (CASES, _complex_rotate_rows, _independent_reuse, _oracle_model, _run_oracle,
                                        _small_gqa)
from tests.test_oracle_pins import _theta_np, mrope_complex, rope_complex

SRC = open(oracle._SRC).read()
rng = np.random.default_rng(99)

MUTANTS = [
    ("rotation sign", "x[ia] = a * c - b * s;", "x[ia] = a * c + b * s;"),
    ("partner update sign", "x[ib] = b * c + a * s;", "x[ib] = b * c - a * s;"),
    ("theta exponent", "pow(base, -2.0 * (double)i / (double)rope_dim)", "pow(base, -1.0 * (double)i / (double)rope_dim)"),
    ("delta sign", "double phi = (double)delta * theta[i];", "double phi = -(double)delta * theta[i];"),
    ("section delta sign", "double phi = (double)deltas[s] * theta[i];", "double phi = (double)deltas[0] * theta[i];"),
    ("section boundary", "if (i >= sections[0]) s = 1;", "if (i > sections[0]) s = 1;"),
    ("V rotated instead of K", "if (channel != 0) return;", "if (channel != 1) return;"),
    ("MLA rotates c_KV", "oracle_rotate_region_sections(row + m->latent_dim,", "oracle_rotate_region_sections(row + 0,"),
    ("patch operand transposed", "acc += u[r] * vmat[(int64_t)j * rank + r];", "acc += u[r] * vmat[(int64_t)r * D + j];"),
    ("patch dropped", "for (int32_t j = 0; j < D; ++j) out[j] += patch[j];",
     "for (int32_t j = 0; j < D; ++j) out[j] += 0.0 * patch[j];"),
    ("frame swapped", "if (m->patch_frame == OR_PATCH_CANONICAL_FRAME) {", "if (m->patch_frame != OR_PATCH_CANONICAL_FRAME) {"),
    ("slot from page index", "return page * page_size + pos % page_size;", "return page * page_size + pos / page_size % page_size;"),
    ("block index off by one", "int64_t blk = pos / page_size;", "int64_t blk = (pos + 1) / page_size;"),
    ("store layer/channel order", "const int64_t sb = store_off[item->chunk_id] + (((int64_t)l * n_ch + ch) * T + t) * D;",
     "const int64_t sb = store_off[item->chunk_id] + (((int64_t)ch * L + l) * T + t) * D;"),
    ("U row shifted", "(int64_t)t * rank;", "(int64_t)(t + 1 < T ? t + 1 : t) * rank;"),
    ("Jacobi rotation sign", "a[(int64_t)k * cols + p] = c * ap - s * aq;", "a[(int64_t)k * cols + p] = c * ap + s * aq;"),
    ("singular values ascending", "if (sigma[k] > sigma[best]) best = k;", "if (sigma[k] < sigma[best]) best = k;"),
    ("orbit mean divisor", "out[e] = s / (double)n;", "out[e] = s / (double)(n + 1);"),
    ("Lloyd centroid sign", "double c = (normal_pdf(t[k]) - normal_pdf(t[k + 1]))",
     "double c = (normal_pdf(t[k + 1]) - normal_pdf(t[k]))"),
    ("Lloyd threshold not a midpoint", "t[k] = 0.5 * (centroids[k - 1] + centroids[k]);",
     "t[k] = 0.5 * (centroids[k] + centroids[k]);"),
    ("K scale step 1/128", "const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    ("K code truncated", "float r = nearbyintf(bf16_bits_to_f32(x[i]) / s);", "float r = truncf(bf16_bits_to_f32(x[i]) / s);"),
    ("Hadamard butterfly sign", "w[j + h] = a - b;", "w[j + h] = b - a;"),
    ("V norm of the transformed row", "acc = fmaf(x[i], x[i], acc);", "acc = fmaf(w[i], w[i], acc);"),
    ("V code of the negated coordinate", "code += (t32[k] <= z) ? 1 : 0;", "code += (t32[k] <= -z) ? 1 : 0;"),
    ("V fields in natural order", "const int32_t bit0 = 6 * (e % half) + (e < half ? 0 : 3);",
     "const int32_t bit0 = 3 * e;"),
    ("Hadamard sign from i|j", "acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -c : c;",
     "acc += (__builtin_popcount((unsigned)(i | j)) & 1) ? -c : c;"),
    ("V decode scaled by 1/sqrt(n)", "out[i] = (double)norm / (double)n * acc;",
     "out[i] = (double)norm / sqrt((double)n) * acc;"),
    ("K scale index transposed", "cs->k_scale[(int64_t)c * m->num_layers + l]", "cs->k_scale[(int64_t)l * cs->n_chunks + c]"),
    ("compressed row order token-major", "const int64_t row = cs->row_offset[c] + (int64_t)l * cs->len[c] + t;",
     "const int64_t row = cs->row_offset[c] + (int64_t)t * m->num_layers + l;"),
    ("interleaved partner taken as rotate-half",
     "int32_t ib = (pairing == OR_INTERLEAVED) ? 2 * i + 1 : i + half;\n    double phi = (double)deltas[s] * theta[i];",
     "int32_t ib = i + half;\n    double phi = (double)deltas[s] * theta[i];"),
    ("head offset by rope_dim", "oracle_rotate_region_sections(row + (int64_t)h * m->head_dim,",
     "oracle_rotate_region_sections(row + (int64_t)h * m->rope_dim,"),
    ("third section boundary", "if (i >= sections[0] + sections[1]) s = 2;", "if (i >= sections[1]) s = 2;"),
    ("theta exponent from a wider row", "theta[i] = pow(base, -2.0 * (double)i / (double)rope_dim);",
     "theta[i] = pow(base, -2.0 * (double)i / (double)(rope_dim + 2));"),
    ("page bound off by one", "if (page < 0 || page >= num_pages) return -1;",
     "if (page < 0 || page > num_pages) return -1;"),
    ("block index bound off by one", "if (blk >= max_pages_per_seq) return -1;",
     "if (blk > max_pages_per_seq) return -1;"),
    ("block-table row stride", "int64_t page = block_table[(int64_t)seq * max_pages_per_seq + blk];",
     "int64_t page = block_table[(int64_t)seq * num_pages + blk];"),
    ("destination offset ignored", "const int64_t pos = item->dst_pos + t;", "const int64_t pos = t;"),
    ("pool layer stride", "const int64_t dst_row = (int64_t)l * num_pages * page_size + dst;",
     "const int64_t dst_row = (int64_t)l * num_pages + dst;"),
    ("V factor read at U's offset",
     "vmat[j * rank + r] = bf16_bits_to_f64(patch[base + ((int64_t)T + j) * rank + r]);",
     "vmat[j * rank + r] = bf16_bits_to_f64(patch[base + ((int64_t)j) * rank + r]);"),
    ("patch layer/channel order",
     "const int64_t base = patch_off[item->patch_id] + ((int64_t)l * n_ch + ch) * (int64_t)(T + D) * rank;",
     "const int64_t base = patch_off[item->patch_id] + ((int64_t)ch * L + l) * (int64_t)(T + D) * rank;"),
    ("chunk length unchecked", "if (store_len[item->chunk_id] != T) { err |= OR_EFLAG_LEN; continue; }", ""),
    ("patch length unchecked", "if (patch_len[item->patch_id] != T) { err |= OR_EFLAG_LEN; continue; }", ""),
    ("patch id bound off by one", "if (item->patch_id >= n_patches) { err |= OR_EFLAG_PATCH_OOB; continue; }",
     "if (item->patch_id > n_patches) { err |= OR_EFLAG_PATCH_OOB; continue; }"),
    ("Jacobi sine not scaled by the cosine", "double s = c * t;", "double s = t;"),
    ("Jacobi stops after one sweep", "if (!rotated) break;", "break;"),
    ("orbit ordering stride", "s += (double)deltas[(int64_t)j * stride + e];",
     "s += (double)deltas[(int64_t)j * n_elems + e];"),
    ("V decode without the norm", "out[i] = (double)norm / (double)n * acc;", "out[i] = 1.0 / (double)n * acc;"),
    ("compressed K taken from V", "const uint16_t* k = store + store_off[c] + ((int64_t)l * 2 + 0) * T * D;",
     "const uint16_t* k = store + store_off[c] + ((int64_t)l * 2 + 1) * T * D;"),
    ("compressed K scale index transposed", "&k_scale[(int64_t)c * L + l]", "&k_scale[(int64_t)l * n_chunks + c]"),
    ("compressed V head offset halved", "oracle_encode_v(v + t * D + (int64_t)h * n, n,",
     "oracle_encode_v(v + t * D + (int64_t)h * (n / 2), n,"),
    ("compressed rows of a layer overlap", "const int64_t row0 = row_offset[c] + (int64_t)l * T;",
     "const int64_t row0 = row_offset[c] + (int64_t)l;"),
    ("in-place relocation writes V too", "const int32_t ch_count = (mode == OR_MODE_RELOCATE_IN_PLACE) ? 1 : n_ch;",
     "const int32_t ch_count = n_ch;"),
    ("in-place patch also rotates", "const int32_t rotate = (mode != OR_MODE_PATCH_IN_PLACE);",
     "const int32_t rotate = 1;"),
    ("in-place patch rewrites unpatched items", "if (mode == OR_MODE_PATCH_IN_PLACE && !use_patch) continue;", ""),
    ("in-place source row without its layer", "src[j] = bf16_bits_to_f64(pin[dst_row * D + j]);",
     "src[j] = bf16_bits_to_f64(pin[dst * D + j]);"),
]


def _build(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    oracle.build(str(c), str(so))
    return oracle.load(str(so))


# ---- independent checks, each raising AssertionError on a mismatch ----------------------------------------

def c_theta(lib):
    np.testing.assert_allclose(oracle.theta(1e6, 128, lib=lib), _theta_np(1e6, 128), rtol=1e-14)


def c_rope(lib):
    for pairing in (oracle.ROTATE_HALF, oracle.INTERLEAVED):
        th = _theta_np(1e4, 64)
        x = rng.standard_normal(64)
        got = oracle.rotate_region(rope_complex(x, 5, th, pairing), th, 1234, pairing, lib=lib)
        np.testing.assert_allclose(got, rope_complex(x, 1239, th, pairing), atol=1e-9)


def c_row(lib):
    m = oracle.model(oracle.GQA, 1, num_kv_heads=2, head_dim=64)
    th = _theta_np(1e4, 64)
    x = rng.standard_normal(128)
    k = oracle.rotate_row(m, th, 0, 77, x, lib=lib)
    for h in range(2):
        np.testing.assert_allclose(k[h * 64:(h + 1) * 64], rope_complex(x[h * 64:(h + 1) * 64], 77, th), atol=1e-11)
    np.testing.assert_array_equal(oracle.rotate_row(m, th, 1, 77, x, lib=lib), x)


def c_mla(lib):
    m = oracle.model(oracle.MLA, 1, rope_dim=64, latent_dim=128)
    th = _theta_np(1e4, 64)
    x = rng.standard_normal(192)
    y = oracle.rotate_row(m, th, 0, 999, x, lib=lib)
    np.testing.assert_array_equal(y[:128], x[:128])
    np.testing.assert_allclose(y[128:], rope_complex(x[128:], 999, th), atol=1e-11)


def c_mrope(lib):
    th = _theta_np(1e6, 128)
    sec = (16, 24, 24)
    x = rng.standard_normal(128)
    got = oracle.rotate_region_sections(mrope_complex(x, (1, 2, 3), th, sec), th, (100, -7, 40), sec, lib=lib)
    np.testing.assert_allclose(got, mrope_complex(x, (101, -5, 43), th, sec), atol=1e-9)


def c_patch(lib):
    m = oracle.model(oracle.GQA, 1, num_kv_heads=2, head_dim=64)
    th = _theta_np(1e4, 64)
    src, u, V = rng.standard_normal(128), rng.standard_normal(8), rng.standard_normal((128, 8))
    np.testing.assert_allclose(oracle.row(m, th, 1, 0, src, u, V, lib=lib), src + V @ u, atol=1e-12)
    want = oracle.rotate_row(m, th, 0, 33, src, lib=lib) + V @ u
    np.testing.assert_allclose(oracle.row(m, th, 0, 33, src, u, V, lib=lib), want, atol=1e-12)


def c_frame(lib):
    ma = oracle.model(oracle.GQA, 1, num_kv_heads=1, head_dim=64)
    mc = oracle.model(oracle.GQA, 1, num_kv_heads=1, head_dim=64, patch_frame=oracle.PATCH_CANONICAL_FRAME)
    th = _theta_np(1e4, 64)
    src, u, V = rng.standard_normal(64), rng.standard_normal(8), rng.standard_normal((64, 8))
    want = rope_complex(src + V @ u, 50, th)
    np.testing.assert_allclose(oracle.row(mc, th, 0, 50, src, u, V, lib=lib), want, atol=1e-11)
    np.testing.assert_allclose(oracle.row(ma, th, 0, 50, src, u, V, lib=lib), rope_complex(src, 50, th) + V @ u,
                               atol=1e-11)


def c_partial(lib):
    m = oracle.model(oracle.GQA, 1, num_kv_heads=2, head_dim=128, rope_dim=64)
    th = _theta_np(1e4, 64)
    x = rng.standard_normal(256)
    k = oracle.rotate_row(m, th, 0, 99, x, lib=lib)
    for h in range(2):
        np.testing.assert_allclose(k[h * 128:h * 128 + 64], rope_complex(x[h * 128:h * 128 + 64], 99, th), atol=1e-11)
        np.testing.assert_array_equal(k[h * 128 + 64:(h + 1) * 128], x[h * 128 + 64:(h + 1) * 128])


def c_slot(lib):
    # several sequences, page ids on and past the bound; the table is the head
    # of a larger array of valid page ids, so that a mutant reading past it
    # reads defined memory and shows up as a wrong slot
    P, n_seqs, mp, num_pages = 16, 3, 5, 20
    full = np.stack([rng.permutation(num_pages)[:mp] for _ in range(40)]).astype(np.int32)
    bt = full[:n_seqs]
    bt[1, 4] = num_pages
    bt[2, 0] = -1
    for seq in range(n_seqs):
        for pos in range(-2, mp * P + 3):
            want = -1
            if 0 <= pos < mp * P:
                page = int(bt[seq, pos // P])
                if 0 <= page < num_pages:
                    want = page * P + pos % P
            assert oracle.slot(bt, mp, num_pages, P, seq, pos, lib=lib) == want


def c_errors(lib):
    wl = _small_gqa()
    n_p = len(wl.patch_lens)

    def run(items, patch_len=None, patch_off=None):
        m = _oracle_model(wl)
        th = oracle.theta(wl.rope_base, wl.rope_dim, lib=lib)
        return oracle.reuse(
            m, th, oracle.MODE_REUSE, store=wl.host_store(), store_off=wl.store_off,
            store_len=np.array(wl.chunk_lens, np.int32), patch=wl.host_patch(),
            patch_off=wl.patch_off if patch_off is None else patch_off,
            patch_len=np.array(wl.patch_lens, np.int32) if patch_len is None else patch_len, rank=wl.rank,
            items=items, block_table=wl.block_table, num_pages=wl.num_pages, page_size=wl.page_size,
            pool_k_in=wl.host_pool(0), pool_v_in=wl.host_pool(1), lib=lib)[0]

    items = wl.items.copy()
    items[0]["n_tokens"] = 69                      # length disagrees with the chunk store only
    plen = np.array(wl.patch_lens, np.int32)
    plen[int(wl.items[0]["patch_id"])] = 69
    assert run(items, patch_len=plen) == oracle.EFLAG_LEN
    plen = np.array(wl.patch_lens, np.int32)
    plen[int(wl.items[0]["patch_id"])] = 71          # length disagrees with the patch store
    assert run(wl.items, patch_len=plen) == oracle.EFLAG_LEN
    items = wl.items.copy()
    items[1]["patch_id"] = n_p                     # one past the last patch; the arrays are views into
    plen = np.append(np.array(wl.patch_lens, np.int32), np.int32(wl.patch_lens[0]))[:n_p]  # longer ones
    poff = np.append(np.asarray(wl.patch_off, np.int64), np.int64(wl.patch_off[0]))[:n_p]
    assert run(items, patch_len=plen, patch_off=poff) == oracle.EFLAG_PATCH_OOB


def c_reuse(lib):
    for case in ("gqa_rank16", "mla_rank8", "gqa_interleaved_canonical"):
        wl = CASES[case]()
        m = _oracle_model(wl)
        th = oracle.theta(wl.rope_base, wl.rope_dim)
        err, pk, pv, wk, wv = oracle.reuse(
            m, th, oracle.MODE_REUSE, store=wl.host_store(), store_off=wl.store_off,
            store_len=np.array(wl.chunk_lens, np.int32), patch=wl.host_patch(), patch_off=wl.patch_off,
            patch_len=np.array(wl.patch_lens, np.int32), rank=wl.rank, items=wl.items, block_table=wl.block_table,
            num_pages=wl.num_pages, page_size=wl.page_size, pool_k_in=wl.host_pool(0),
            pool_v_in=wl.host_pool(1) if wl.n_ch == 2 else None, lib=lib)
        ik, iv, iwk, iwv = _independent_reuse(wl)
        np.testing.assert_array_equal(wk.astype(bool), iwk)
        np.testing.assert_allclose(pk[iwk], ik[iwk], atol=1e-10)
        if wl.n_ch == 2:
            np.testing.assert_allclose(pv[iwv], iv[iwv], atol=1e-10)


def c_inplace(lib):
    # sliding-window survival: K of the survivors' pages turned by delta, V and other pages untouched
    wl = W.sliding_window(num_layers=2, n_resident=6, n_evict=2, T=32, page_size=16, num_kv_heads=2)
    k_in, v_in = wl.host_pool(0), wl.host_pool(1)
    err, pk, pv, wk, wv = _run_oracle(wl, k_in, v_in, lib=lib)
    assert err == 0 and not wv.any()
    np.testing.assert_array_equal(pv, oracle.bf16_bits_to_f64(v_in))
    kin = oracle.bf16_bits_to_f64(k_in)
    surv = set(wl.block_table[0].tolist())
    theta = _theta_np(wl.rope_base, 128)
    for layer in range(2):
        for page in range(wl.num_pages):
            if page in surv:
                want = _complex_rotate_rows(kin[layer, page], 2, 128, 128, 0, -64, theta, W.ROTATE_HALF)
                np.testing.assert_allclose(pk[layer, page], want, atol=1e-10)
            else:
                np.testing.assert_array_equal(pk[layer, page], kin[layer, page])
    # patch in place: U V^T added with no rotation; an item without a patch is not written
    wl = _small_gqa().replace(mode="apply_patch", pool_init="random", chunk_lens=[])
    wl.items["patch_id"][0] = -1
    k_in, v_in = wl.host_pool(0), wl.host_pool(1)
    err, pk, pv, wk, wv = _run_oracle(wl, k_in, v_in, lib=lib)
    assert err == 0
    for it_i, it in enumerate(wl.items):
        pos = int(it["dst_pos"]) + np.arange(int(it["n_tokens"]))
        pages, slots = wl.block_table[0, pos // 16], pos % 16
        assert wk[:, pages, slots].all() == (it_i != 0) and wv[:, pages, slots].all() == (it_i != 0)
        if it_i == 0:
            continue
        p = int(it["patch_id"])
        for layer in range(wl.num_layers):
            for ch, img, src in ((0, pk, k_in), (1, pv, v_in)):
                U = oracle.bf16_bits_to_f64(wl.u_rows(p, layer, ch))
                V = oracle.bf16_bits_to_f64(wl.v_rows(p, layer, ch))
                want = oracle.bf16_bits_to_f64(src[layer, pages, slots]) + U @ V.T
                np.testing.assert_allclose(img[layer, pages, slots], want, atol=1e-12)


def c_svd(lib):
    a = rng.standard_normal((30, 10))
    us, v, sig = oracle.jacobi_svd(a, lib=lib)
    np.testing.assert_allclose(sig, np.linalg.svd(a, compute_uv=False), rtol=1e-10)
    np.testing.assert_allclose(us @ v.T, a, atol=1e-10)


def c_orbit(lib):
    d = rng.standard_normal((4, 50)).astype(np.float32)
    np.testing.assert_allclose(oracle.orbit_mean(d, lib=lib), d.astype(np.float64).mean(axis=0), atol=1e-15)
    # orderings further apart than the elements averaged (stride 40, 25 elements)
    full = rng.standard_normal((3, 40)).astype(np.float32)
    out = np.zeros(25, np.float64)
    lib.oracle_orbit_mean(oracle._ptr(full), 3, 40, 25, oracle._ptr(out))
    np.testing.assert_allclose(out, full[:, :25].astype(np.float64).mean(axis=0), atol=1e-15)


def c_codebook(lib):
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "lloyd_max_gaussian_n8.json")))
    c32, t32 = oracle.v_codebook(lib=lib)
    np.testing.assert_allclose(c32[4:], g["positive_outputs"], atol=g["abs_tol"])
    np.testing.assert_allclose(t32[3:], g["positive_thresholds"][:4], atol=g["abs_tol"])


def c_kquant(lib):
    x = gen.f32_to_bf16_bits(rng.standard_normal(300).astype(np.float32) * 2)
    xf = oracle.bf16_bits_to_f64(x)
    q, s = oracle.quantize_k(x, lib=lib)
    assert np.abs(q).max() == 127
    assert np.all(np.abs(xf - q.astype(np.float64) * s) <= 0.5 * s * (1 + 1e-5))


def c_vcodec(lib):
    n = 128
    c32, t32 = oracle.v_codebook(lib=lib)
    Hm = linalg.hadamard(n).astype(np.float64)
    codes = rng.integers(0, 8, n)
    got = oracle.decode_v(_pack(codes)[None], np.array([2.0], np.float32), n, lib=lib)[0]
    np.testing.assert_allclose(got, 2.0 / n * (Hm @ c32[codes].astype(np.float64)), atol=1e-12)
    x = gen.f32_to_bf16_bits(rng.standard_normal((4, n)).astype(np.float32))
    packed, norms = oracle.encode_v(x, lib=lib)
    xf = oracle.bf16_bits_to_f64(x)
    for r in range(4):
        assert abs(norms[r] - np.linalg.norm(xf[r])) <= 1e-6 * np.linalg.norm(xf[r])
        z = Hm @ xf[r] / np.linalg.norm(xf[r])
        near = np.abs(z[:, None] - c32[None, :].astype(np.float64)).argmin(axis=1)
        tie = np.min(np.abs(z[:, None] - t32[None, :].astype(np.float64)), axis=1) < 1e-5
        assert np.all((_unpack(packed[r], n) == near) | tie)


def c_reuse_comp(lib):
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=20, rank=8, page_size=16)
    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim)
    r = wl.random_compressed()
    cs = oracle.Compressed(r["k_codes"], r["k_scale"], r["v_codes"], r["v_norm"], r["row_offset"], r["len"],
                           oracle.v_codebook(lib=lib)[0])
    th = oracle.theta(wl.rope_base, wl.rope_dim, lib=lib)
    err, pk, pv, wk, wv = oracle.reuse_compressed(
        m, th, cs, patch=wl.host_patch(), patch_off=wl.patch_off, patch_len=np.array(wl.patch_lens, np.int32),
        rank=wl.rank, items=wl.items, block_table=wl.block_table, num_pages=wl.num_pages, page_size=wl.page_size,
        pool_k_in=wl.host_pool(0), pool_v_in=wl.host_pool(1), lib=lib)
    ik, iv, iwk, iwv = _independent_reuse_compressed(wl, cs)
    np.testing.assert_array_equal(wk.astype(bool), iwk)
    np.testing.assert_allclose(pk[iwk], ik[iwk], atol=1e-10)
    np.testing.assert_allclose(pv[iwv], iv[iwv], atol=1e-10)


def c_compress(lib):
    wl = W.gqa_video(num_layers=2, n_chunks=2, T=12, rank=0, page_size=16)
    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim)
    check_store_encoding(wl, oracle.compress_store(m, wl.host_store(), wl.store_off,
                                                    np.array(wl.chunk_lens, np.int32), lib=lib))


CHECKS = [c_theta, c_rope, c_row, c_partial, c_mla, c_mrope, c_patch, c_frame, c_slot, c_errors, c_reuse, c_inplace, c_svd,
          c_orbit, c_codebook, c_kquant, c_vcodec, c_compress, c_reuse_comp]


def test_unmutated_oracle_passes_every_check(tmp_path):
    lib = _build(tmp_path, "clean", SRC)
    for check in CHECKS:
        check(lib)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_every_planted_mistake_is_caught(tmp_path, name, old, new):
    assert SRC.count(old) == 1, f"mutation site not unique: {old}"
    lib = _build(tmp_path, name.replace(" ", "_").replace("/", "_"), SRC.replace(old, new))
    failed = []
    for check in CHECKS:
        try:
            check(lib)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no check caught the mutant '{name}'"
