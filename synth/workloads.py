"""Workload shapes for the Kamera reuse operator and their seeded fills.

Each workload is a batch of reuse items over a canonical chunk store, a patch
store and a paged KV pool, with the shapes of the workloads the Kamera page
describes (video-frame chunks of about a thousand tokens, GQA and MLA
backbones, ranks 8-64, Kamera §3 window operations).  Values are synthetic
and seeded (``synth.gen``); no dataset or model weights are involved.

Layouts (shared by the CUDA path and the oracle, bf16 bit patterns):
  chunk store  per chunk c at element offset store_off[c]: [layer][channel][T_c][D]
  patch store  per patch p at element offset patch_off[p]:
               [layer][channel] ( U [T_p][rank] then V [D][rank] )
  pool         K and V each [layer][num_pages][page_size][D]   (MLA: K only)
  block table  [n_seqs][max_pages_per_seq] int32 page ids
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

from . import gen

MHA, GQA, MLA = 0, 1, 2
ROTATE_HALF, INTERLEAVED = 0, 1
AFTER_ROTATION, CANONICAL_FRAME = 0, 1

ITEM_DTYPE = np.dtype(
    [("chunk_id", np.int32), ("patch_id", np.int32), ("delta", np.int64), ("seq", np.int32),
     ("n_tokens", np.int32), ("dst_pos", np.int64)],
    align=True,
)

SENTINEL_BITS = 0xFFFF  # a bf16 NaN: marks pool slots that must stay untouched


@dataclass
class Workload:
    name: str
    family: int
    num_layers: int
    num_kv_heads: int = 0
    head_dim: int = 0
    rope_dim: int = 0
    latent_dim: int = 0
    rope_base: float = 10000.0
    pairing: int = ROTATE_HALF
    patch_frame: int = AFTER_ROTATION
    mode: str = "reuse"  # "reuse" | "relocate_in_place" | "apply_patch"
    chunk_lens: list = field(default_factory=list)
    rank: int = 0
    patch_lens: list = field(default_factory=list)
    items: np.ndarray = None
    page_size: int = 64
    num_pages: int = 0
    block_table: np.ndarray = None
    seed: int = 1
    sigma_kv: float = 1.0
    sigma_uv: float = 0.02
    outlier_permille: int = 0
    outlier_sigma: float = 8.0
    pool_init: str = "sentinel"  # "sentinel" | "random"
    rope_sections: tuple = (0, 0, 0)  # M-RoPE pairs per (temporal, height, width) section; zeros = plain RoPE
    section_deltas: np.ndarray = None  # [n_items][3] per-section shifts (None: the item's delta everywhere)
    inv_freq: np.ndarray = None  # explicit fp64 frequency table [rope_dim/2] (None: rope_base^(-2i/rope_dim))

    # ---- derived shapes ----------------------------------------------------
    def __post_init__(self):
        if self.family != MLA and self.rope_dim == 0:
            self.rope_dim = self.head_dim

    @property
    def D(self) -> int:
        return self.latent_dim + self.rope_dim if self.family == MLA else self.num_kv_heads * self.head_dim

    @property
    def n_ch(self) -> int:
        return 1 if self.family == MLA else 2

    @property
    def store_off(self) -> np.ndarray:
        sizes = [self.num_layers * self.n_ch * t * self.D for t in self.chunk_lens]
        return np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64) if sizes else np.zeros(0, np.int64)

    @property
    def store_elems(self) -> int:
        return int(sum(self.num_layers * self.n_ch * t * self.D for t in self.chunk_lens))

    @property
    def patch_off(self) -> np.ndarray:
        sizes = [self.num_layers * self.n_ch * (t + self.D) * self.rank for t in self.patch_lens]
        return np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64) if sizes else np.zeros(0, np.int64)

    @property
    def patch_elems(self) -> int:
        return int(sum(self.num_layers * self.n_ch * (t + self.D) * self.rank for t in self.patch_lens))

    @property
    def pool_shape(self) -> tuple:
        return (self.num_layers, self.num_pages, self.page_size, self.D)

    @property
    def tokens(self) -> int:
        """Reused tokens per call (each token counted once across all layers)."""
        return int(np.maximum(self.items["n_tokens"], 0).sum())

    def algorithmic_bytes(self) -> int:
        """Bytes one call must move at minimum: every reused row read and
        written once per layer and channel, plus the patch factors once."""
        L, D = self.num_layers, self.D
        total = 0
        for it in self.items:
            T = int(it["n_tokens"])
            if self.mode == "relocate_in_place":
                total += L * T * D * 2 * 2  # K rows only, read + write
                continue
            total += L * self.n_ch * T * D * 2 * 2
            if self.rank > 0 and it["patch_id"] >= 0:
                total += L * self.n_ch * (T + D) * self.rank * 2
        return total

    def patch_flops(self) -> int:
        if self.rank == 0 or self.mode == "relocate_in_place":
            return 0
        n = sum(int(it["n_tokens"]) for it in self.items if it["patch_id"] >= 0)
        return 2 * self.rank * n * self.D * self.n_ch * self.num_layers

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    # ---- counter-stream seeds --------------------------------------------------
    def stream(self, tag: int) -> int:
        return gen.stream_id(self.seed, tag)

    def _slab(self, layer: int, ch: int) -> int:
        return layer * self.n_ch + ch

    # ---- host (numpy) generation, any slice --------------------------------------
    def store_rows(self, chunk: int, layer: int, ch: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
        """Canonical rows [t1 - t0][D] of (chunk, layer, channel) as bf16 bits."""
        t1 = self.chunk_lens[chunk] if t1 is None else t1
        return gen.fill_rows(self.stream(gen.STREAM_KV), t1 - t0, self.D, gen.kv_index(chunk, layer, ch, t0, 0),
                             1 << gen.D_BITS, gen.scale_f32(self.sigma_kv), self.stream(gen.STREAM_OUTLIER),
                             gen.outlier_key(layer, ch), gen.scale_f32(self.outlier_sigma), self.outlier_permille)

    def u_rows(self, patch: int, layer: int, ch: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
        t1 = self.patch_lens[patch] if t1 is None else t1
        return gen.fill_rows(self.stream(gen.STREAM_U), t1 - t0, self.rank, gen.u_index(patch, layer, ch, t0, 0),
                             1 << gen.R_BITS, gen.scale_f32(self.sigma_uv))

    def v_rows(self, patch: int, layer: int, ch: int) -> np.ndarray:
        return gen.fill_rows(self.stream(gen.STREAM_V), self.D, self.rank, gen.v_index(patch, layer, ch, 0, 0),
                             1 << gen.R_BITS, gen.scale_f32(self.sigma_uv))

    def pool_rows(self, ch: int, layer: int, page: int) -> np.ndarray:
        """Initial rows [P][D] of one pool page (random init only)."""
        tag = gen.STREAM_POOL if ch == 0 else gen.STREAM_POOL + 100
        return gen.fill_rows(self.stream(tag), self.page_size, self.D, gen.pool_index(layer, page, 0, 0),
                             1 << gen.D_BITS, gen.scale_f32(self.sigma_kv))

    def host_store(self) -> np.ndarray:
        out = np.zeros(self.store_elems, np.uint16)
        for c, T in enumerate(self.chunk_lens):
            base = int(self.store_off[c])
            for layer in range(self.num_layers):
                for ch in range(self.n_ch):
                    o = base + self._slab(layer, ch) * T * self.D
                    out[o:o + T * self.D] = self.store_rows(c, layer, ch).reshape(-1)
        return out

    def host_patch(self) -> np.ndarray:
        out = np.zeros(self.patch_elems, np.uint16)
        m, D = self.rank, self.D
        for p, T in enumerate(self.patch_lens):
            base = int(self.patch_off[p])
            for layer in range(self.num_layers):
                for ch in range(self.n_ch):
                    o = base + self._slab(layer, ch) * (T + D) * m
                    out[o:o + T * m] = self.u_rows(p, layer, ch).reshape(-1)
                    out[o + T * m:o + (T + D) * m] = self.v_rows(p, layer, ch).reshape(-1)
        return out

    def host_pool(self, ch: int) -> np.ndarray:
        shape = self.pool_shape
        if self.pool_init == "sentinel":
            return np.full(shape, SENTINEL_BITS, np.uint16)
        out = np.zeros(shape, np.uint16)
        for layer in range(self.num_layers):
            for page in range(self.num_pages):
                out[layer, page] = self.pool_rows(ch, layer, page)
        return out

    # ---- compressed canonical store (int8 K, 3-bit V; PolyKV §2B) ----------------------
    @property
    def comp_row_offset(self) -> np.ndarray:
        """Chunks back to back: chunk c, layer l, token t is row comp_row_offset[c] + l*T_c + t."""
        sizes = [self.num_layers * t for t in self.chunk_lens]
        return np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64) if sizes else np.zeros(0, np.int64)

    @property
    def comp_rows(self) -> int:
        return int(sum(self.num_layers * t for t in self.chunk_lens))

    def random_compressed(self) -> dict:
        """A compressed store filled with seeded random contents (any byte is a
        valid code): K codes uniform in [-127, 127], V code bytes uniform,
        per-(chunk, layer) K scales and per-head-row V norms uniform around
        the bf16 store's scale."""
        rows, D, H, n, L = self.comp_rows, self.D, self.num_kv_heads, self.head_dim, self.num_layers
        kb = gen.random_bytes(self.stream(gen.STREAM_KCODE), rows * D)
        k_codes = ((kb.astype(np.int32) % 255) - 127).astype(np.int8).reshape(rows, D)
        v_codes = gen.random_bytes(self.stream(gen.STREAM_VCODE), rows * H * (3 * n // 8)).reshape(rows, H, -1)
        nc = len(self.chunk_lens)
        k_scale = gen.uniform_f32(self.stream(gen.STREAM_KSCALE), np.arange(nc * L, dtype=np.uint64),
                                  0.5 * 4 * self.sigma_kv / 127, 1.5 * 4 * self.sigma_kv / 127).reshape(nc, L)
        v_norm = gen.uniform_f32(self.stream(gen.STREAM_VNORM), np.arange(rows * H, dtype=np.uint64),
                                 0.5 * self.sigma_kv * np.sqrt(n), 1.5 * self.sigma_kv * np.sqrt(n)).reshape(rows, H)
        return dict(k_codes=k_codes, k_scale=k_scale, v_codes=v_codes, v_norm=v_norm,
                    row_offset=self.comp_row_offset, len=np.array(self.chunk_lens, np.int32))

    def compressed_bytes(self) -> int:
        """Bytes one call must move at minimum when the canonical rows come
        from the compressed store: K codes (1 byte/value) and V codes (3/8
        byte/value) plus one V norm per head row read once, the bf16 output
        rows written once, and the patch factors read once."""
        L, D, H = self.num_layers, self.D, self.num_kv_heads
        total = 0
        for it in self.items:
            T = int(it["n_tokens"])
            total += L * T * (D + 3 * D // 8 + 4 * H) + L * 2 * T * D * 2
            if self.rank > 0 and it["patch_id"] >= 0:
                total += L * 2 * (T + D) * self.rank * 2
        return total

    # ---- device fills (CUDA twin of the generator) ----------------------------------
    def device_store(self, torch, device="cuda"):
        from . import device as dev
        buf = torch.empty(max(self.store_elems, 8), dtype=torch.bfloat16, device=device)
        slab_stride_idx = (2 // self.n_ch) << (gen.T_BITS + gen.D_BITS)
        for c, T in enumerate(self.chunk_lens):
            dev.fill_rows(buf.data_ptr() + 2 * int(self.store_off[c]), n_slabs=self.num_layers * self.n_ch, rows=T,
                          row_len=self.D, out_slab_stride=T * self.D, out_row_stride=self.D,
                          stream=self.stream(gen.STREAM_KV), idx0=gen.kv_index(c, 0, 0, 0, 0),
                          idx_slab_stride=slab_stride_idx, idx_row_stride=1 << gen.D_BITS,
                          scale=float(gen.scale_f32(self.sigma_kv)), outlier_stream=self.stream(gen.STREAM_OUTLIER),
                          okey0=gen.outlier_key(0, 0), okey_slab_stride=(2 // self.n_ch) << gen.D_BITS,
                          outlier_scale=float(gen.scale_f32(self.outlier_sigma)),
                          outlier_permille=self.outlier_permille,
                          cuda_stream=torch.cuda.current_stream().cuda_stream)
        return buf

    def device_patch(self, torch, device="cuda"):
        from . import device as dev
        buf = torch.empty(max(self.patch_elems, 8), dtype=torch.bfloat16, device=device)
        m, D = self.rank, self.D
        if m == 0:
            return buf
        cs = torch.cuda.current_stream().cuda_stream
        for p, T in enumerate(self.patch_lens):
            base = buf.data_ptr() + 2 * int(self.patch_off[p])
            dev.fill_rows(base, n_slabs=self.num_layers * self.n_ch, rows=T, row_len=m, out_slab_stride=(T + D) * m,
                          out_row_stride=m, stream=self.stream(gen.STREAM_U), idx0=gen.u_index(p, 0, 0, 0, 0),
                          idx_slab_stride=(2 // self.n_ch) << (gen.T_BITS + gen.R_BITS),
                          idx_row_stride=1 << gen.R_BITS, scale=float(gen.scale_f32(self.sigma_uv)), cuda_stream=cs)
            dev.fill_rows(base + 2 * T * m, n_slabs=self.num_layers * self.n_ch, rows=D, row_len=m,
                          out_slab_stride=(T + D) * m, out_row_stride=m, stream=self.stream(gen.STREAM_V),
                          idx0=gen.v_index(p, 0, 0, 0, 0),
                          idx_slab_stride=(2 // self.n_ch) << (gen.D_BITS + gen.R_BITS),
                          idx_row_stride=1 << gen.R_BITS, scale=float(gen.scale_f32(self.sigma_uv)), cuda_stream=cs)
        return buf

    def device_pool(self, torch, ch: int, device="cuda"):
        from . import device as dev
        L, NP, P, D = self.pool_shape
        buf = torch.empty((L, NP, P, D), dtype=torch.bfloat16, device=device)
        if self.pool_init == "sentinel":
            buf.view(torch.int16).fill_(-1)  # 0xFFFF
            return buf
        tag = gen.STREAM_POOL if ch == 0 else gen.STREAM_POOL + 100
        cs = torch.cuda.current_stream().cuda_stream
        for layer in range(L):
            dev.fill_rows(buf.data_ptr() + 2 * layer * NP * P * D, n_slabs=NP, rows=P, row_len=D,
                          out_slab_stride=P * D, out_row_stride=D, stream=self.stream(tag),
                          idx0=gen.pool_index(layer, 0, 0, 0), idx_slab_stride=1 << (8 + gen.D_BITS),
                          idx_row_stride=1 << gen.D_BITS, scale=float(gen.scale_f32(self.sigma_kv)), cuda_stream=cs)
        return buf


# ---- helpers ------------------------------------------------------------------------

def make_items(chunk_ids, patch_ids, deltas, seqs, lens, dst_pos) -> np.ndarray:
    n = np.broadcast(np.asarray(chunk_ids), np.asarray(patch_ids), np.asarray(deltas), np.asarray(seqs),
                     np.asarray(lens), np.asarray(dst_pos)).size
    it = np.zeros(n, ITEM_DTYPE)
    it["chunk_id"], it["patch_id"], it["delta"] = chunk_ids, patch_ids, deltas
    it["seq"], it["n_tokens"], it["dst_pos"] = seqs, lens, dst_pos
    return it


def shuffled_block_table(seed: int, n_seqs: int, pages_per_seq: int, num_pages: int | None = None) -> np.ndarray:
    """Each sequence gets pages_per_seq distinct pages of a seeded shuffle of the pool."""
    num_pages = num_pages or n_seqs * pages_per_seq
    perm = gen.permutation(gen.stream_id(seed, gen.STREAM_PERM), num_pages)
    return perm[: n_seqs * pages_per_seq].reshape(n_seqs, pages_per_seq).astype(np.int32)


def _random_deltas(seed: int, n: int, lo: int = -32768, hi: int = 32768) -> np.ndarray:
    return gen.uniform_int(gen.stream_id(seed, gen.STREAM_DELTA), np.arange(n, dtype=np.uint64), lo, hi)


# ---- the five workload shapes ----------------------------------------------------------

def with_mrope(wl: Workload, sections=(16, 24, 24), seed: int | None = None) -> Workload:
    """M-RoPE variant (the temporal / height / width split of Qwen2-VL-style
    multimodal RoPE): a seeded temporal shift and a separate spatial shift
    (shared by height and width) per item."""
    seed = wl.seed if seed is None else seed
    n = len(wl.items)
    dt = _random_deltas(seed + 11, n)
    ds = _random_deltas(seed + 12, n)
    sd = np.stack([dt, ds, ds], axis=1).astype(np.int64)
    return wl.replace(rope_sections=tuple(sections), section_deltas=sd, name=wl.name + "_mrope")


def tiny_mha(seed: int = 0x4B414D45 + 1) -> Workload:
    """MHA, 1 layer, 4 heads x 64, one 256-token chunk, rank 8, delta 1000,
    base 1e4, rotate-half, output into a contiguous [T][H][d] buffer (one
    256-slot page, identity block table)."""
    T = 256
    items = make_items([0], [0], [1000], [0], [T], [0])
    return Workload("tiny_mha", MHA, 1, num_kv_heads=4, head_dim=64, rope_base=1e4, chunk_lens=[T], rank=8,
                    patch_lens=[T], items=items, page_size=T, num_pages=1,
                    block_table=np.zeros((1, 1), np.int32), seed=seed)


def gqa_video(seed: int = 0x4B414D45 + 2, num_layers: int = 28, n_chunks: int = 16, T: int = 1024,
              rank: int = 32, page_size: int = 64) -> Workload:
    """GQA shaped like Qwen2.5-VL-7B: 28 layers, 4 KV heads x 128, base 1e6;
    16 chunks x 1024 tokens, 1 % outlier channels x8, rank-32 patch per layer
    per K/V, delta uniform in [-32768, 32768], one sequence, shuffled pages."""
    n_pos = n_chunks * T
    ppseq = -(-n_pos // page_size)
    items = make_items(np.arange(n_chunks), np.arange(n_chunks) if rank else -1, _random_deltas(seed, n_chunks),
                       0, T, np.arange(n_chunks) * T)
    return Workload("gqa_video", GQA, num_layers, num_kv_heads=4, head_dim=128, rope_base=1e6,
                    chunk_lens=[T] * n_chunks, rank=rank, patch_lens=[T] * n_chunks if rank else [], items=items,
                    page_size=page_size, num_pages=ppseq, block_table=shuffled_block_table(seed, 1, ppseq),
                    seed=seed, outlier_permille=10)


def mla_lite(seed: int = 0x4B414D45 + 3, num_layers: int = 27, n_chunks: int = 8, T: int = 2048, rank: int = 16,
             page_size: int = 64) -> Workload:
    """MLA shaped like DeepSeek-V2-Lite: 27 layers, c_KV 512 + k_rope 64;
    8 chunks x 2048 tokens, only k_rope re-rotated, c_KV copied byte for byte,
    rank-16 patch on the whole latent row (V rows split 512 + 64)."""
    n_pos = n_chunks * T
    ppseq = -(-n_pos // page_size)
    items = make_items(np.arange(n_chunks), np.arange(n_chunks) if rank else -1, _random_deltas(seed, n_chunks),
                       0, T, np.arange(n_chunks) * T)
    return Workload("mla_lite", MLA, num_layers, rope_dim=64, latent_dim=512, rope_base=1e4,
                    chunk_lens=[T] * n_chunks, rank=rank, patch_lens=[T] * n_chunks if rank else [], items=items,
                    page_size=page_size, num_pages=ppseq, block_table=shuffled_block_table(seed, 1, ppseq),
                    seed=seed)


def sliding_window(seed: int = 0x4B414D45 + 4, num_layers: int = 32, n_resident: int = 64, n_evict: int = 8,
                   T: int = 1024, page_size: int = 64, num_kv_heads: int = 8) -> Workload:
    """Sliding-window survival, GQA 8B-shaped (32 layers, 8 KV heads x 128,
    base 5e5): 64 resident chunks x 1024 tokens in the pool; the 8 oldest are
    evicted and the 56 survivors are re-rotated in place by -8192 (no patch).
    The survivors keep their pages; their block-table row is shifted so that
    they now start at position 0."""
    pages_per_chunk = T // page_size
    num_pages = n_resident * pages_per_chunk
    old_table = shuffled_block_table(seed, 1, num_pages)  # positions before the slide
    new_table = old_table[:, n_evict * pages_per_chunk:].copy()
    n_surv = n_resident - n_evict
    delta = -n_evict * T
    items = make_items(-1, -1, delta, 0, T, np.arange(n_surv) * T)
    return Workload("sliding_window", GQA, num_layers, num_kv_heads=num_kv_heads, head_dim=128, rope_base=5e5,
                    mode="relocate_in_place", items=items, page_size=page_size, num_pages=num_pages,
                    block_table=new_table, seed=seed, pool_init="random")


def long_video(seed: int = 0x4B414D45 + 5, num_layers: int = 32, n_reorder: int = 128, n_recall: int = 32,
               T: int = 1296, rank: int = 64, page_size: int = 64, num_kv_heads: int = 8) -> Workload:
    """Long-video reorder + recall, GQA 8B-shaped: a store of 160 chunks x 1296
    tokens; a seeded permutation places chunks 0..127 at positions pi(c)*1296
    with their shared orbit patches (rank 64), then the 32 evicted chunks
    128..159 are recalled after them with fresh rank-64 patches.  Chunks start
    mid-page (1296 = 20.25 pages).  delta = new position (the canonical chunk
    is stored at position 0)."""
    n = n_reorder + n_recall
    perm = gen.permutation(gen.stream_id(seed, gen.STREAM_PERM + 1), n_reorder)
    dst = np.concatenate([perm * T, (n_reorder + np.arange(n_recall)) * T]).astype(np.int64)
    n_pos = n * T
    ppseq = -(-n_pos // page_size)
    items = make_items(np.arange(n), np.arange(n), dst, 0, T, dst)
    return Workload("long_video", GQA, num_layers, num_kv_heads=num_kv_heads, head_dim=128, rope_base=5e5,
                    chunk_lens=[T] * n, rank=rank, patch_lens=[T] * n, items=items, page_size=page_size,
                    num_pages=ppseq, block_table=shuffled_block_table(seed, 1, ppseq), seed=seed)


WORKLOADS = {
    "tiny_mha": tiny_mha,
    "gqa_video": gqa_video,
    "mla_lite": mla_lite,
    "sliding_window": sliding_window,
    "long_video": long_video,
}
