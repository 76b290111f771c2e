"""Glue for the GPU tests, the smoke check and the benchmark: seeded workload ->
device tensors -> one call through the C ABI -> host readback, and the
comparison rule against the fp64 oracle.

Comparison rule (on rotated and/or patched K/V):
    |gpu - ref| <= ulp_bf16(ref) + 1e-3,   ulp_bf16(x) = 2^(floor(log2|x|) - 7)
Kamera §3 states the production hook rebuilds the cache "within bf16
rounding"; one bf16 ulp of the exact value plus an absolute 1e-3 for values
near zero is that statement made testable.  Unpatched, unrotated columns (MLA
c_KV, V with no patch, delta = 0 without patch) and every untouched slot must
be bit-identical.
"""
from __future__ import annotations

import numpy as np

import position_invariant_kv_kamera_gb300 as pk
from synth import workloads as W

ABS_TOL = 1e-3


def model_for(wl: W.Workload, t: dict | None = None):
    return pk.model_desc(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim, wl.latent_dim,
                         wl.pairing, wl.patch_frame, wl.rope_base, inv_freq=wl.inv_freq,
                         rope_sections=wl.rope_sections, section_delta=(t or {}).get("section_delta"))


def device_inputs(wl: W.Workload, torch, device="cuda", pool_host=None, with_store=True) -> dict:
    """All device tensors of one call; the pool is the sentinel / seeded initial pool.
    with_store=False leaves out the bf16 chunk store (a compressed store serves instead)."""
    t = {}
    if wl.mode == "reuse" and with_store:
        t["store"] = wl.device_store(torch, device)
        t["store_off"] = torch.tensor(wl.store_off, dtype=torch.int64, device=device)
        t["store_len"] = torch.tensor(np.array(wl.chunk_lens, np.int32), dtype=torch.int32, device=device)
    if wl.rank and wl.mode != "relocate_in_place":
        t["patch"] = wl.device_patch(torch, device)
        t["patch_off"] = torch.tensor(wl.patch_off, dtype=torch.int64, device=device)
        t["patch_len"] = torch.tensor(np.array(wl.patch_lens, np.int32), dtype=torch.int32, device=device)
    items = np.ascontiguousarray(wl.items.astype(pk.REUSE_ITEM))
    t["items"] = torch.from_numpy(items.view(np.uint8).copy()).to(device)
    t["block_table"] = torch.from_numpy(np.ascontiguousarray(wl.block_table, np.int32)).to(device)
    if pool_host is not None:
        t["pool_k"] = torch.from_numpy(pool_host[0].view(np.int16)).to(device).view(torch.bfloat16)
        t["pool_v"] = (torch.from_numpy(pool_host[1].view(np.int16)).to(device).view(torch.bfloat16)
                       if wl.n_ch == 2 else None)
    else:
        t["pool_k"] = wl.device_pool(torch, 0, device)
        t["pool_v"] = wl.device_pool(torch, 1, device) if wl.n_ch == 2 else None
    t["err"] = torch.zeros(1, dtype=torch.int32, device=device)
    if wl.section_deltas is not None:
        t["section_delta"] = torch.from_numpy(np.ascontiguousarray(wl.section_deltas, np.int64)).to(device)
    return t


def call(wl: W.Workload, t: dict, mode: str | None = None, stream=None, raise_on_error=True) -> int:
    mode = mode or wl.mode
    return pk.call(mode, model_for(wl, t), items=t["items"], pool_k=t["pool_k"], pool_v=t["pool_v"],
                   block_table=t["block_table"], page_size=wl.page_size, store=t.get("store"),
                   store_off=t.get("store_off"), store_len=t.get("store_len"), patch=t.get("patch"),
                   patch_off=t.get("patch_off"), patch_len=t.get("patch_len"),
                   rank=wl.rank if "patch" in t else 0, err_flag=t["err"], stream=stream,
                   raise_on_error=raise_on_error)


def to_bits(x) -> np.ndarray:
    """bf16 device tensor -> host uint16 bit patterns."""
    return x.view(__import__("torch").int16).cpu().numpy().view(np.uint16)


def bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def within_tol(gpu_f64: np.ndarray, ref: np.ndarray) -> np.ndarray:
    return np.abs(gpu_f64 - ref) <= ulp_bf16(ref) + ABS_TOL


def oracle_theta(wl: W.Workload) -> np.ndarray:
    """The frequency table both sides use: the workload's explicit table, or
    the oracle's ladder rope_base^(-2i/rope_dim)."""
    import oracle

    if wl.inv_freq is not None:
        return np.ascontiguousarray(wl.inv_freq, np.float64)
    return oracle.theta(wl.rope_base, wl.rope_dim)


def oracle_reference(wl: W.Workload, pool_k_in=None, pool_v_in=None):
    """fp64 oracle over the whole workload (small workloads only)."""
    import oracle

    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim, wl.latent_dim,
                     wl.pairing, wl.patch_frame, wl.rope_sections)
    th = oracle_theta(wl)
    mode = {"reuse": oracle.MODE_REUSE, "relocate": oracle.MODE_REUSE,
            "relocate_in_place": oracle.MODE_RELOCATE_IN_PLACE, "apply_patch": oracle.MODE_PATCH_IN_PLACE}[wl.mode]
    pk_in = wl.host_pool(0) if pool_k_in is None else pool_k_in
    pv_in = (wl.host_pool(1) if pool_v_in is None else pool_v_in) if wl.n_ch == 2 else None
    kw = {}
    if wl.mode in ("reuse", "relocate"):
        kw.update(store=wl.host_store(), store_off=wl.store_off, store_len=np.array(wl.chunk_lens, np.int32))
    if wl.rank and wl.mode != "relocate_in_place":
        kw.update(patch=wl.host_patch(), patch_off=wl.patch_off, patch_len=np.array(wl.patch_lens, np.int32),
                  rank=wl.rank)
    return oracle.reuse(m, th, mode, items=wl.items, block_table=wl.block_table, num_pages=wl.num_pages,
                        page_size=wl.page_size, pool_k_in=pk_in, pool_v_in=pv_in, section_deltas=wl.section_deltas,
                        **kw)


def compare_pool(gpu_bits: np.ndarray, in_bits: np.ndarray, ref: np.ndarray, wrote: np.ndarray,
                 exact_cols: slice | None = None) -> dict:
    """Element-wise comparison of one pool channel against the oracle image.

    Untouched rows must equal the input bits; written rows must be within the
    tolerance (and bit-exact on ``exact_cols`` when given)."""
    wrote = wrote.astype(bool)
    report = {"rows_written": int(wrote.sum())}
    untouched_ok = np.array_equal(gpu_bits[~wrote], in_bits[~wrote])
    report["untouched_bit_exact"] = bool(untouched_ok)
    g = bits_to_f64(gpu_bits[wrote])
    r = ref[wrote]
    ok = within_tol(g, r)
    report["within_tol"] = bool(ok.all())
    report["n_bad"] = int((~ok).sum())
    report["max_abs_err"] = float(np.abs(g - r).max()) if g.size else 0.0
    if exact_cols is not None and g.size:
        report["exact_cols_bit_exact"] = bool(np.array_equal(g[..., exact_cols], r[..., exact_cols]))
    return report


def assert_report(rep: dict):
    assert rep["untouched_bit_exact"], rep
    assert rep["within_tol"], rep
    if "exact_cols_bit_exact" in rep:
        assert rep["exact_cols_bit_exact"], rep


# ---- compressed canonical store (PolyKV §2B) ---------------------------------------------------

COMP_KEYS = ("k_codes", "k_scale", "v_codes", "v_norm", "row_offset", "len")


def comp_arrays(cs) -> dict:
    """Host arrays of a compressed store: from the oracle's encoder
    (``oracle.Compressed``) or from ``Workload.random_compressed()``."""
    if isinstance(cs, dict):
        return {k: cs[k] for k in COMP_KEYS}
    return {"k_codes": cs.k_codes, "k_scale": cs.k_scale, "v_codes": cs.v_codes, "v_norm": cs.v_norm,
            "row_offset": cs.row_offset, "len": cs.len}


def oracle_store(arrs: dict):
    """The same host arrays as the oracle's store object (with the oracle's codebook)."""
    import oracle

    c32, _ = oracle.v_codebook()
    return oracle.Compressed(arrs["k_codes"], arrs["k_scale"], arrs["v_codes"], arrs["v_norm"], arrs["row_offset"],
                             arrs["len"], c32)


def device_compressed(arrs: dict, torch, device="cuda"):
    """(kamera_compressed_store, device tensors) for host arrays."""
    t = {k: torch.from_numpy(np.ascontiguousarray(arrs[k])).to(device) for k in COMP_KEYS}
    return pk.compressed_store(t["k_codes"], t["k_scale"], t["v_codes"], t["v_norm"], t["row_offset"], t["len"]), t


def empty_compressed(wl: W.Workload, torch, device="cuda"):
    """A device compressed store of the workload's row layout, to be filled by the encoder."""
    rows, D, H, n = wl.comp_rows, wl.D, wl.num_kv_heads, wl.head_dim
    t = {"k_codes": torch.zeros((rows, D), dtype=torch.int8, device=device),
         "k_scale": torch.zeros((len(wl.chunk_lens), wl.num_layers), dtype=torch.float32, device=device),
         "v_codes": torch.zeros((rows, H, 3 * n // 8), dtype=torch.uint8, device=device),
         "v_norm": torch.zeros((rows, H), dtype=torch.float32, device=device),
         "row_offset": torch.from_numpy(wl.comp_row_offset).to(device),
         "len": torch.from_numpy(np.array(wl.chunk_lens, np.int32)).to(device)}
    return pk.compressed_store(t["k_codes"], t["k_scale"], t["v_codes"], t["v_norm"], t["row_offset"], t["len"]), t


def call_compressed(wl: W.Workload, t: dict, cstore, stream=None, raise_on_error=True) -> int:
    return pk.call_compressed(model_for(wl, t), cstore, items=t["items"], pool_k=t["pool_k"], pool_v=t["pool_v"],
                              block_table=t["block_table"], page_size=wl.page_size, patch=t.get("patch"),
                              patch_off=t.get("patch_off"), patch_len=t.get("patch_len"),
                              rank=wl.rank if "patch" in t else 0, err_flag=t["err"], stream=stream,
                              raise_on_error=raise_on_error)


def oracle_reference_compressed(wl: W.Workload, ocs, pool_k_in=None, pool_v_in=None):
    """fp64 oracle of the reuse operator reading the compressed store ``ocs``."""
    import oracle

    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim, wl.latent_dim,
                     wl.pairing, wl.patch_frame, wl.rope_sections)
    th = oracle_theta(wl)
    kw = {}
    if wl.rank:
        kw.update(patch=wl.host_patch(), patch_off=wl.patch_off, patch_len=np.array(wl.patch_lens, np.int32),
                  rank=wl.rank)
    return oracle.reuse_compressed(m, th, ocs, items=wl.items, block_table=wl.block_table, num_pages=wl.num_pages,
                                   page_size=wl.page_size,
                                   pool_k_in=wl.host_pool(0) if pool_k_in is None else pool_k_in,
                                   pool_v_in=wl.host_pool(1) if pool_v_in is None else pool_v_in,
                                   section_deltas=wl.section_deltas, **kw)
