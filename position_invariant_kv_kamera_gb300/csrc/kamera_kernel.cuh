// kamera_kernel.cuh -- the fused Kamera reuse kernel for sm_103a.
//
// One persistent, warp-specialised kernel computes, for every reuse item,
// layer, channel and token (Kamera: Unified Position-Invariant Multimodal KV
// Cache for Training-Free Reuse, §2 reuse equation):
//
//     out = R(delta) . KV(B|empty) + U_m V_m^T        -> bf16 -> paged pool slot
//
// Row block: 128 destination positions (aligned to 128 in position space) of
// one (item, layer, channel); it splits into n_cb tiles of BN columns.  CTAs
// take work units round-robin: whole row blocks for as many full rounds as
// the grid allows (their per-row-block set-up -- page segments, phase table --
// serves all n_cb tiles), then the row blocks of the partial last round split
// into single tiles, so that round is one tile deep and calls with fewer row
// blocks than CTAs spread over as many SMs as they have tiles.  Per CTA
// (384 threads, one CTA per SM):
//   warp 0      TMA producer: the canonical tile (64-column boxes, 128B
//               swizzle; from the chunk store, or page by page from the pool
//               for the in-place modes) into a ring of shared-memory stages.
//   warp 1      owns TMEM; one lane issues tcgen05.mma (M=128, N=BN, K=16
//               steps): P = U . V^T into an fp32 TMEM accumulator, two buffers.
//   warp 2      TMA store issuer: whole page segments of the finished tile go
//               to the pool with cp.async.bulk.tensor stores (8-row boxes for
//               the in-item part of partly covered pages).
//   warp 11     TMA producer of the patch factors: the U tile [128 x m] and
//               the V tile [BN x m] of each tile, in K chunks of m / ksplit,
//               as whole chunk rows swizzled at their width (K-major), or --
//               rank 8 and the compressed variant -- as 16-byte core matrices
//               (rank 8 with a zeroed second K group), into slots.
//   warps 3-10  epilogue, two warps per TMEM lane quadrant, each half taking
//               half of the tile's rotation units: tcgen05.ld the patch row,
//               rotate the key row's RoPE pairs by delta*theta_i (fp64 angle
//               reduction, fp32 sincos and math), add, round to bf16 in place;
//               the few edge rows of partly covered pages that do not fill an
//               8-row box are stored by their own threads.
// Compressed canonical store (kComp; PolyKV, gist.science summary, §2B): the
// producer stages int8 K codes (128-column boxes, 128B swizzle) or packed 3-bit
// V codes behind the stage's bf16 output tile, and the epilogue decodes them
// on the fly -- K: code * per-(chunk, layer) scale; V: each 6-bit field
// (codes i and i + d/2) becomes x_i +- x_{i+d/2} by one lookup in a
// lane-replicated table of centroid sums, then a Walsh-Hadamard transform of
// length d/2 in registers and the scale ||v|| / d.  Each epilogue half decodes
// its half of every head.  The decoded row then takes the same rotation,
// patch and store as a bf16 canonical row.
// Every wait on an mbarrier is bounded (2 s unless the call sets another
// limit): on expiry the kernel sets
// KAMERA_EFLAG_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "kamera.h"
#include "ptx.cuh"

namespace kamera {

constexpr int BM = 128;             // tile rows = TMEM lanes = M of the MMA
constexpr int NUM_WARPS = 12;
constexpr int NUM_THREADS = 32 * NUM_WARPS;
constexpr int EPI_WARP0 = 3;        // first epilogue warp
constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = 32 * EPI_WARPS;
constexpr int UV_WARP = 11;         // loads the patch factors
constexpr int MAX_GROUPS = 64;      // 32-column groups per row (D <= 2048)
constexpr int MAX_PAIRS = 128;      // rope_dim / 2
constexpr int BOX_COLS = 64;        // 64 bf16 = one 128-byte swizzle row
constexpr uint32_t BOX_BYTES = BM * 128;  // one 64-column box of 128 rows
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // default bound of every wait (the call may set another)

// group kinds (per 32-column group of a key row); a positive value is a
// rotate-half first half whose partner group is that many groups to the right
constexpr int8_t GK_PLAIN = 0;
constexpr int8_t GK_SECOND = -1;
constexpr int8_t GK_INTERLEAVED = -2;

struct Params {
  CUtensorMap src_map;      // chunk store as rows [rows][D]: box 64 x 128, 128B swizzle
  CUtensorMap pool_map[2];  // pool K / V as rows [L*pages*P][D]: box 64 x S (S = min(P,128)), 128B swizzle
  CUtensorMap pool_map8[2]; // the same with 8-row boxes, for partly covered page segments
  CUtensorMap u_map;        // patch store: rows [rows][m], box (m/ksplit, 128), swizzled; rank 8: (8, rows, 1)
  CUtensorMap v_map;        // the same with BN-row boxes
  const kamera_reuse_item* items;
  int32_t n_items;
  int32_t src_pool;  // 0: gather from the chunk store, 1: in place from the pool
  const int64_t* store_off;
  const int32_t* store_len;
  int64_t store_elems;
  int32_t n_chunks;
  int32_t has_patches;
  const int64_t* patch_off;
  const int32_t* patch_len;
  int64_t patch_elems;
  int32_t n_patches;
  int32_t rank;
  int32_t ksplit;      // patch factors staged in this many K chunks per tile
  int32_t ksteps;      // K=16 MMA steps per chunk: ceil(rank / ksplit / 16)
  int32_t kg_alloc;    // 8-element K groups held in smem per operand row and chunk (>= 2)
  int32_t uv_row_bytes;  // bytes of one operand row of a chunk, swizzled at that width (32/64/128);
                         // 0: rank 8, K-major core matrices with a zeroed second K group
  int32_t need_patch;  // items without a patch have no work (patch-only mode)
  uint16_t* pool[2];
  int64_t num_pages;
  int32_t page_size;
  int32_t page_shift;
  const int32_t* block_table;
  int32_t n_seqs;
  int32_t max_pages;
  int32_t num_layers;
  int32_t D;
  int32_t n_ch_layout;  // channels in the store / patch layout (2, MLA 1)
  int32_t n_ch_work;    // channels processed (in-place relocate: keys only)
  int32_t BN;
  int32_t n_cb;      // column blocks processed per row
  int32_t cb_first;  // first processed column block
  int32_t stages;     // canonical tile stages
  int32_t uv_slots;   // patch-factor slots (U and V tiles)
  int32_t seg_rows;   // rows per pool page segment in a tile (min(P, 128))
  int32_t seg_shift;  // log2(seg_rows)
  int32_t rotate;    // rotate channel 0
  int32_t frame;     // kamera_patch_frame
  int32_t n_pairs;
  int32_t sec_end0, sec_end1;      // M-RoPE: pairs [0, sec_end0) section 0, [sec_end0, sec_end1) section 1, rest 2
  const int64_t* section_delta;    // [n_items][3] per-section shifts, or nullptr (every section: item delta)
  uint32_t stage_bytes, u_bytes, v_bytes, tmem_cols;  // stage_bytes = one canonical tile
  int32_t* err_flag;
  uint64_t wait_limit_ns;  // bound of every wait
  int32_t test_unarm;      // test only: the producer leaves its first stage unfilled (the waits on it run out)
  // compressed canonical store (kComp)
  CUtensorMap kc_map;  // K codes as rows [rows][D] uint8: box 128 x 128, 128B swizzle
  CUtensorMap vc_map;  // V codes as rows [rows][3D/8] uint8: box 3BN/8 x 128, no swizzle
  const int64_t* comp_row_offset;  // [n_chunks]: chunk c, layer l, token t at row offset[c] + l*T + t
  const int32_t* comp_len;         // [n_chunks]
  const float* k_scale;            // [n_chunks][num_layers]
  const float* v_norm;             // [rows][D / head_dim]
  int64_t comp_rows;
  int32_t head_dim;
  uint32_t out_bytes;    // bf16 output tile at the start of each stage; the codes follow it
  uint32_t table_bytes;  // the replicated centroid-sum table
  float pair_sum[64];    // c[a] + c[b] at index a + 8b (fp32 codebook)
  int8_t group_kind[MAX_GROUPS];
  uint8_t pair_base[MAX_GROUPS];
  uint8_t owner0[MAX_GROUPS];  // epilogue half that processes the unit starting at group g (rotated tiles)
  double theta[MAX_PAIRS];
};

// ---- work decomposition ---------------------------------------------------------------

struct Walker {
  int32_t item;
  int64_t base, count;
  int64_t dst_pos;
  int64_t d0, d1, d2;  // the item's shift of each M-RoPE section (all equal without sections)
  int32_t T, seq, chunk, patch;
  uint32_t n_tb;
};

// Row blocks of item i (0 if it is skipped); fills the walker's item fields.
// Error bits are collected in err (the caller decides whether to report them).
__device__ __forceinline__ int64_t item_tiles(const Params& p, int32_t i, Walker& w, int32_t& err) {
  const kamera_reuse_item it = p.items[i];
  w.T = it.n_tokens;
  w.seq = it.seq;
  w.chunk = it.chunk_id;
  w.patch = -1;
  w.dst_pos = it.dst_pos;
  w.d0 = w.d1 = w.d2 = it.delta;
  if (p.section_delta) {
    w.d0 = p.section_delta[(int64_t)i * 3 + 0];
    w.d1 = p.section_delta[(int64_t)i * 3 + 1];
    w.d2 = p.section_delta[(int64_t)i * 3 + 2];
  }
  w.n_tb = 0;
  if (it.n_tokens == 0) return 0;
  if (it.n_tokens < 0 || it.dst_pos < 0) { err |= KAMERA_EFLAG_LEN; return 0; }
  if (it.seq < 0 || it.seq >= p.n_seqs) { err |= KAMERA_EFLAG_PAGE_OOB; return 0; }
  const int64_t T = it.n_tokens;
  if (p.comp_row_offset) {
    if (it.chunk_id < 0 || it.chunk_id >= p.n_chunks) { err |= KAMERA_EFLAG_CHUNK_OOB; return 0; }
    if (p.comp_len[it.chunk_id] != it.n_tokens) { err |= KAMERA_EFLAG_LEN; return 0; }
    const int64_t r0 = p.comp_row_offset[it.chunk_id];
    if (r0 < 0 || r0 + (int64_t)p.num_layers * T > p.comp_rows) { err |= KAMERA_EFLAG_CHUNK_OOB; return 0; }
  } else if (!p.src_pool) {
    if (it.chunk_id < 0 || it.chunk_id >= p.n_chunks) { err |= KAMERA_EFLAG_CHUNK_OOB; return 0; }
    if (p.store_len[it.chunk_id] != it.n_tokens) { err |= KAMERA_EFLAG_LEN; return 0; }
    const int64_t off = p.store_off[it.chunk_id];
    if (off < 0 || off % p.D != 0 || off + (int64_t)p.num_layers * p.n_ch_layout * T * p.D > p.store_elems) {
      err |= KAMERA_EFLAG_CHUNK_OOB;
      return 0;
    }
  }
  if (p.has_patches && it.patch_id >= 0) {
    if (it.patch_id >= p.n_patches) { err |= KAMERA_EFLAG_PATCH_OOB; return 0; }
    if (p.patch_len[it.patch_id] != it.n_tokens) { err |= KAMERA_EFLAG_LEN; return 0; }
    const int64_t off = p.patch_off[it.patch_id];
    if (off < 0 || off % p.rank != 0 ||
        off + (int64_t)p.num_layers * p.n_ch_layout * (T + p.D) * p.rank > p.patch_elems) {
      err |= KAMERA_EFLAG_PATCH_OOB;
      return 0;
    }
    w.patch = it.patch_id;
  }
  if (p.need_patch && w.patch < 0) return 0;
  w.n_tb = (uint32_t)((it.dst_pos + T + BM - 1) / BM - it.dst_pos / BM);
  const int64_t count = (int64_t)p.num_layers * p.n_ch_work * w.n_tb;
  if (count > (int64_t)0xFFFFFFFF) { err |= KAMERA_EFLAG_LEN; return 0; }  // the decode is 32-bit
  return count;
}

__device__ __forceinline__ void walker_init(Walker& w) {
  w.item = -1;
  w.base = 0;
  w.count = 0;
}

// Advance (monotonically) to the item holding global row block g.
__device__ __forceinline__ void walk_to(const Params& p, Walker& w, int64_t g) {
  while (g >= w.base + w.count) {
    w.base += w.count;
    ++w.item;
    int32_t e = 0;
    w.count = item_tiles(p, w.item, w, e);
  }
}

struct Tile {
  int32_t layer, ch, cb;
  int64_t pos0;  // destination position of tile row 0
};

// Row block g of the walker's item (order: layer, channel, token block); an
// item has fewer than 2^32 row blocks, so the decode runs in 32 bits.  The
// column block is filled in by the caller's inner loop.
__device__ __forceinline__ Tile decode(const Params& p, const Walker& w, int64_t g) {
  const uint32_t local = (uint32_t)(g - w.base);
  Tile t;
  const uint32_t q = local / w.n_tb;
  const uint32_t tb = local - q * w.n_tb;
  const uint32_t nch = (uint32_t)p.n_ch_work;
  t.layer = (int32_t)(q / nch);
  t.ch = (int32_t)(q - (uint32_t)t.layer * nch);
  t.cb = p.cb_first;
  t.pos0 = (w.dst_pos & ~(int64_t)(BM - 1)) + (int64_t)tb * BM;
  return t;
}

// Work unit u < full_rb + tail_tiles of the schedule: units [0, full_rb) are
// whole row blocks, the rest single tiles of the remaining row blocks (tile tt
// of them is column block tt mod n_cb of row block full_rb + tt / n_cb).  The
// tail holds fewer than gridDim.x * n_cb tiles, so its index fits 32 bits.
struct Unit {
  int64_t rb;
  int cb0, cb1;  // column blocks [cb0, cb1) relative to cb_first
};

__device__ __forceinline__ Unit unit_of(int64_t u, int64_t full_rb, int n_cb) {
  Unit x;
  if (u < full_rb) {
    x.rb = u;
    x.cb0 = 0;
    x.cb1 = n_cb;
  } else {
    const uint32_t tt = (uint32_t)(u - full_rb), q = tt / (uint32_t)n_cb;
    x.rb = full_rb + q;
    x.cb0 = (int)(tt - q * (uint32_t)n_cb);
    x.cb1 = x.cb0 + 1;
  }
  return x;
}

// A page segment of a tile (rows [sg*S, sg*S + S)): its pool row, or -1 when
// its page is out of range.  `full` = every row of the segment belongs to the item.
struct Segment {
  int32_t y;
  bool full, any;
};

__device__ __forceinline__ Segment segment(const Params& p, const Walker& w, const Tile& t, int sg) {
  Segment s;
  const int64_t ps = t.pos0 + (int64_t)sg * p.seg_rows;
  s.any = !(ps + p.seg_rows <= w.dst_pos || ps >= w.dst_pos + w.T);
  s.full = ps >= w.dst_pos && ps + p.seg_rows <= w.dst_pos + w.T;
  s.y = -1;
  if (!s.any) return s;
  const int64_t blk = ps >> p.page_shift;
  if (blk >= p.max_pages) return s;
  const int32_t page = p.block_table[(int64_t)w.seq * p.max_pages + blk];
  if (page < 0 || page >= p.num_pages) return s;
  s.y = (int32_t)(((int64_t)t.layer * p.num_pages + page) * p.page_size + (ps & (p.page_size - 1)));
  return s;
}

// ---- shared memory ---------------------------------------------------------------------

struct SmemMisc {
  uint32_t tmem_base;
  int32_t abort_flag;
  int64_t full_rb;     // row blocks dealt whole: the full rounds of the grid
  int64_t tail_tiles;  // tiles of the remaining row blocks, dealt one by one
  uint64_t wait_limit;  // ns
};

struct Smem {
  uint8_t* stages;     // stage s at stages + s * stage_bytes
  uint8_t* uv;         // slot u at uv + u * (u_bytes + v_bytes): U tile then V tile
  float* table;        // compressed V: pair_sum[e] for lane l at table[e * 32 + l]
  uint64_t* full;      // [stages] TMA loads landed
  uint64_t* uv_full;   // [uv_slots] patch factors landed
  uint64_t* uv_empty;  // [uv_slots] slot free (MMA done with it)
  uint64_t* empty;     // [stages] stage free (8 epilogue warps + the store warp)
  uint64_t* computed;  // [stages] tile computed in place (8 epilogue warps)
  uint64_t* tfull;     // [2] accumulator ready
  uint64_t* tempty;    // [2] accumulator drained
  uint64_t* drain;     // [1]
  SmemMisc* misc;
  float2* cs;        // [2][n_pairs_pad] phase tables, one per row-block parity: per two pairs (c, c', s, s')
};

__device__ __forceinline__ Smem carve_smem(uint8_t* raw, const Params& p) {
  const uint32_t a = smem_addr(raw);
  uint8_t* base = raw + ((1024u - (a & 1023u)) & 1023u);
  Smem s;
  s.stages = base;
  s.uv = base + (size_t)p.stages * p.stage_bytes;
  s.table = reinterpret_cast<float*>(s.uv + (size_t)p.uv_slots * (p.u_bytes + p.v_bytes));
  uint8_t* q = reinterpret_cast<uint8_t*>(s.table) + p.table_bytes;
  s.full = reinterpret_cast<uint64_t*>(q);
  s.empty = s.full + p.stages;
  s.computed = s.empty + p.stages;
  s.uv_full = s.computed + p.stages;
  s.uv_empty = s.uv_full + p.uv_slots;
  s.tfull = s.uv_empty + p.uv_slots;
  s.tempty = s.tfull + 2;
  s.drain = s.tempty + 2;
  s.misc = reinterpret_cast<SmemMisc*>(s.drain + 1);
  const uintptr_t cs_at = (reinterpret_cast<uintptr_t>(s.misc) + 32 + 15) & ~uintptr_t(15);
  s.cs = reinterpret_cast<float2*>(cs_at);
  return s;
}

// rows of one phase table: the rope pairs, rounded up to a float4 multiple
__host__ __device__ constexpr int pairs_pad(int n_pairs) { return (n_pairs + 1) & ~1; }

__host__ __device__ constexpr uint32_t smem_extra_bytes(int stages, int uv_slots, int n_pairs) {
  return 1024 /*alignment slack*/ + 8u * (3u * stages + 2u * uv_slots + 5u) + 32u + 16u +
         8u * 2u * (uint32_t)pairs_pad(n_pairs);
}

// Bounded wait.  Returns false on abort (another role gave up) or on expiry
// (then it raises the abort flag and the timeout error bit).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, SmemMisc* misc, int32_t* err_flag,
                                             bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns(), limit = misc->wait_limit;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *reinterpret_cast<volatile int32_t*>(&misc->abort_flag)) return false;
    if (global_timer_ns() - t0 > limit) {
      *reinterpret_cast<volatile int32_t*>(&misc->abort_flag) = 1;
      if (err_flag) atomicOr(err_flag, KAMERA_EFLAG_TIMEOUT);
      return false;
    }
  }
}

// ---- epilogue helpers ----------------------------------------------------------------------

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// cos/sin of delta*theta_i: the angle is formed and reduced modulo 2*pi in fp64
// (two-constant Cody-Waite reduction), then sin/cos are taken in fp32.
__device__ __forceinline__ float2 phase_cs(int64_t delta, double theta) {
  const double kTwoPiHi = 6.283185307179586;       // fp64 nearest to 2*pi
  const double kTwoPiLo = 2.4492935982947064e-16;  // 2*pi - kTwoPiHi
  const double kInvTwoPi = 0.15915494309189535;    // 1 / (2*pi)
  const double phi = (double)delta * theta;
  const double k = rint(phi * kInvTwoPi);
  double r = fma(-k, kTwoPiHi, phi);
  r = fma(-k, kTwoPiLo, r);
  float s, c;
  sincosf((float)r, &s, &c);
  return make_float2(c, s);
}

// Row view of a 128B-swizzled tile: 16-byte chunk j (8 columns) of this row.
struct RowView {
  uint32_t base;  // tile base + row * 128
  uint32_t sw;    // row & 7
  __device__ __forceinline__ uint32_t chunk(int col) const {
    return base + (uint32_t)(col >> 6) * BOX_BYTES + ((((uint32_t)col >> 3) & 7u) ^ sw) * 16u;
  }
};

// Results of 16 columns at tile column c: back into the tile (for the TMA
// store) and, for rows of partly covered pages, straight to the pool row.
__device__ __forceinline__ void put16(uint32_t a0, uint32_t a1, uint4 v0, uint4 v1, uint16_t* gdst, int c) {
  sts128(a0, v0);
  sts128(a1, v1);
  if (gdst) {
    stg128_cs(gdst + c, v0);
    stg128_cs(gdst + c + 8, v1);
  }
}

// int8 codes -> fp32 pairs: a byte permute builds the float 2^23 + (q + 128),
// the subtraction of 2^23 + 128 is exact, and the product with the scale is
// the one rounding (the same value as (float)q * scale).
__device__ __forceinline__ void dequant16(uint4 v, float scale, float2* x) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
  const float2 bias = make_float2(8388736.0f, 8388736.0f), sc = make_float2(scale, scale);
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int b = 0; b < 4; b += 2) {
      const float2 f = make_float2(__uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7540u | (uint32_t)b)),
                                   __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7540u | (uint32_t)(b + 1))));
      x[2 * k + b / 2] = mul_f2(sub_f2(f, bias), sc);
    }
}

__device__ __forceinline__ void unpack8_f2(uint4 v, float2* x) {
  x[0] = make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u));
  x[1] = make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
  x[2] = make_float2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u));
  x[3] = make_float2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
}

__device__ __forceinline__ uint4 pack8_f2(const float2* x) {
  return make_uint4(pack2(x[0].x, x[0].y), pack2(x[1].x, x[1].y), pack2(x[2].x, x[2].y), pack2(x[3].x, x[3].y));
}

__device__ __forceinline__ float2 acc_f2(const uint32_t* acc, int e) {
  return make_float2(__uint_as_float(acc[2 * e]), __uint_as_float(acc[2 * e + 1]));
}

// Canonical values of this thread's row, 16 columns at a time, as 8 pairs of
// neighbouring columns.
struct SrcTile {  // the bf16 tile itself (TMA-loaded canonical rows)
  RowView rv;
  __device__ __forceinline__ void load16(int c, float2* x) const {
    const uint4 v0 = lds128(rv.chunk(c)), v1 = lds128(rv.chunk(c + 8));
    unpack8_f2(v0, x);
    unpack8_f2(v1, x + 4);
  }
};
struct SrcK8 {  // int8 K codes: 128-column boxes, 128B swizzle, one scale per (chunk, layer)
  uint32_t base;  // staging + row * 128
  uint32_t sw;    // row & 7
  float scale;
  __device__ __forceinline__ void load16(int c, float2* x) const {
    dequant16(lds128(base + (uint32_t)(c >> 7) * BOX_BYTES + ((((uint32_t)c >> 4) & 7u) ^ sw) * 16u), scale, x);
  }
};

// 16 columns without rotation: out = x + P (patched); without a patch the
// bf16 tile already holds the output and only a thread-stored row is copied
// out (a compressed source is always decoded and written).
template <bool kPatched, bool kComp, class Src>
__device__ __forceinline__ void epi_plain16(const Src& src, const RowView& rv, int c0, uint32_t taddr,
                                            uint16_t* gdst) {
  const uint32_t a0 = rv.chunk(c0), a1 = rv.chunk(c0 + 8);
  if (!kPatched && !kComp) {
    if (gdst) {
      stg128_cs(gdst + c0, lds128(a0));
      stg128_cs(gdst + c0 + 8, lds128(a1));
    }
    return;
  }
  uint32_t acc[16];
  if (kPatched) tmem_ld16(taddr + (uint32_t)c0, acc);
  float2 x[8];
  src.load16(c0, x);
  if (kPatched) {
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = add_f2(x[e], acc_f2(acc, e));
  }
  put16(a0, a1, pack8_f2(x), pack8_f2(x + 4), gdst, c0);
}

// 16 rotate-half pairs (cA + e, cB + e), pair index pb + e, two pairs per
// paired operation:  a' = a cos - b sin,  b' = b cos + a sin.
template <bool kPatched, bool kCanonicalFrame, class Src>
__device__ __forceinline__ void epi_rotate16(const Src& src, const RowView& rv, int cA, int cB, int pb,
                                             uint32_t taddr, const float2* cs, uint16_t* gdst) {
  uint32_t accA[16], accB[16];
  if (kPatched) {
    tmem_ld16(taddr + (uint32_t)cA, accA);
    tmem_ld16(taddr + (uint32_t)cB, accB);
  }
  float2 xa[8], xb[8];
  src.load16(cA, xa);
  src.load16(cB, xb);
  if (kPatched) tmem_ld_wait();
  const float4* cs4 = reinterpret_cast<const float4*>(cs + pb);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float4 t = cs4[e];  // (cos, cos', sin, sin') of pairs pb + 2e and pb + 2e + 1
    const float2 c = make_float2(t.x, t.y), sn = make_float2(t.z, t.w);
    float2 a = xa[e], b = xb[e];
    if (kPatched && kCanonicalFrame) {
      a = add_f2(a, acc_f2(accA, e));
      b = add_f2(b, acc_f2(accB, e));
    }
    float2 ra = sub_f2(mul_f2(a, c), mul_f2(b, sn));
    float2 rb = fma_f2(a, sn, mul_f2(b, c));
    if (kPatched && !kCanonicalFrame) {
      ra = add_f2(ra, acc_f2(accA, e));
      rb = add_f2(rb, acc_f2(accB, e));
    }
    xa[e] = ra;
    xb[e] = rb;
  }
  put16(rv.chunk(cA), rv.chunk(cA + 8), pack8_f2(xa), pack8_f2(xa + 4), gdst, cA);
  put16(rv.chunk(cB), rv.chunk(cB + 8), pack8_f2(xb), pack8_f2(xb + 4), gdst, cB);
}

// 8 interleaved pairs (2e, 2e+1) in 16 columns, pair index pb + e.
template <bool kPatched, bool kCanonicalFrame, class Src>
__device__ __forceinline__ void epi_interleaved16(const Src& src, const RowView& rv, int c0, int pb, uint32_t taddr,
                                                  const float2* cs, uint16_t* gdst) {
  uint32_t acc[16];
  if (kPatched) tmem_ld16(taddr + (uint32_t)c0, acc);
  float2 x[8];  // x[e] = (a, b) of pair pb + e
  src.load16(c0, x);
  if (kPatched) tmem_ld_wait();
  const float4* cs4 = reinterpret_cast<const float4*>(cs + pb);
#pragma unroll
  for (int e2 = 0; e2 < 4; ++e2) {
    const float4 t = cs4[e2];  // (cos, cos', sin, sin') of pairs pb + 2*e2 and pb + 2*e2 + 1
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = 2 * e2 + h;
      const float c = h ? t.y : t.x, s = h ? t.w : t.z;
      float a = x[e].x, b = x[e].y;
      if (kPatched && kCanonicalFrame) {
        a += __uint_as_float(acc[2 * e]);
        b += __uint_as_float(acc[2 * e + 1]);
      }
      float ra = fmaf(a, c, -b * s);
      float rb = fmaf(b, c, a * s);
      if (kPatched && !kCanonicalFrame) {
        ra += __uint_as_float(acc[2 * e]);
        rb += __uint_as_float(acc[2 * e + 1]);
      }
      x[e] = make_float2(ra, rb);
    }
  }
  put16(rv.chunk(c0), rv.chunk(c0 + 8), pack8_f2(x), pack8_f2(x + 4), gdst, c0);
}

// One tile row's share of the compute phase for epilogue half h.  gdst: the
// pool row (at the tile's first column) when this row is stored by its
// threads, else nullptr.
template <bool kPatched, bool kCanonicalFrame, bool kComp, class Src>
__device__ __forceinline__ void epi_row(const Params& p, const Src& src, const RowView& rv, int cb, bool rot, int h,
                                        uint32_t taddr, const float2* cs, uint16_t* gdst) {
  if (!kPatched && !kComp && !rot && !gdst) return;  // bit copy of the whole tile: nothing to do
  const int ng = p.BN / 32;
  const int g0 = cb * ng;
  for (int gl = 0; gl < ng; ++gl) {
    const int g = g0 + gl;
    const int8_t kind = rot ? p.group_kind[g] : GK_PLAIN;
    if (kind == GK_SECOND) continue;
    const int owner = rot ? p.owner0[g] : (gl & 1);
    if (owner != h) continue;
    const int c0 = gl * 32;
    if (kind == GK_PLAIN) {
      epi_plain16<kPatched, kComp>(src, rv, c0, taddr, gdst);
      epi_plain16<kPatched, kComp>(src, rv, c0 + 16, taddr, gdst);
    } else if (kind == GK_INTERLEAVED) {
      const int pb = p.pair_base[g];
      epi_interleaved16<kPatched, kCanonicalFrame>(src, rv, c0, pb, taddr, cs, gdst);
      epi_interleaved16<kPatched, kCanonicalFrame>(src, rv, c0 + 16, pb + 8, taddr, cs, gdst);
    } else {
      const int pb = p.pair_base[g];
      const int cB = (gl + kind) * 32;
      epi_rotate16<kPatched, kCanonicalFrame>(src, rv, c0, cB, pb, taddr, cs, gdst);
      epi_rotate16<kPatched, kCanonicalFrame>(src, rv, c0 + 16, cB + 16, pb + 16, taddr, cs, gdst);
    }
  }
}

// ---- compressed V: Walsh-Hadamard decode ----------------------------------------------------

// In-place unnormalised Walsh-Hadamard transform of N values (Sylvester
// order) held as N/2 pairs v[k] = (u[2k], u[2k+1]): the stride-1 butterflies
// inside each pair, then every wider stride on whole pairs with paired adds.
template <int N>
__device__ __forceinline__ void fwht_pairs(float2* v) {
#pragma unroll
  for (int k = 0; k < N / 2; ++k) v[k] = make_float2(v[k].x + v[k].y, v[k].x - v[k].y);
#pragma unroll
  for (int h = 1; h < N / 2; h <<= 1)
#pragma unroll
    for (int i = 0; i < N / 2; i += 2 * h)
#pragma unroll
      for (int k = i; k < i + h; ++k) {
        const float2 a = v[k], b = v[k + h];
        v[k] = add_f2(a, b);
        v[k + h] = sub_f2(a, b);
      }
}

// Bit k of a head row's code stream is set in this mask iff it is one of the
// upper three bits of its 6-bit field; XOR-ing it turns every field (a, b)
// into (a, 7 - b), i.e. c[b] into c[7 - b] = -c[b].
__host__ __device__ constexpr uint32_t upper_field_mask(int word) {
  uint32_t m = 0;
  for (int b = 0; b < 32; ++b)
    if (((word * 32 + b) % 6) >= 3) m |= 1u << b;
  return m;
}

// Half h of one head of this thread's row: outputs j = h*HD/2 + i, i < HD/2,
//     v^_j = (||v|| / HD) * (H_{HD/2} (x_lo +- x_hi))_i,
// where x_lo / x_hi are the centroids of codes i and i + HD/2 (field i) and
// the sign is + for h = 0, - for h = 1 (the first butterfly of H_HD).
//   codes: shared address of the head's packed codes (3*HD/8 bytes)
//   scale: ||v|| / HD;   c_out: tile column of output i = 0
//   tab_lane: shared address of the pair table + 4 * lane
//   patched: add the patch accumulator (warp-uniform)
template <int HD>
__device__ __forceinline__ void epi_vhalf(const RowView& rv, uint32_t codes, float scale, int h, int c_out,
                                          uint32_t taddr, uint32_t tab_lane, uint16_t* gdst, bool patched) {
  constexpr int NW = 3 * HD / 32;  // 32-bit code words per head row
  constexpr int NF = HD / 2;       // fields = outputs of this half
  uint32_t w[NW];
  if (HD == 128) {
#pragma unroll
    for (int k = 0; k < NW / 4; ++k) {
      const uint4 v = lds128(codes + 16u * k);
      w[4 * k] = v.x;
      w[4 * k + 1] = v.y;
      w[4 * k + 2] = v.z;
      w[4 * k + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < NW / 2; ++k) {
      const uint2 v = lds64(codes + 8u * k);
      w[2 * k] = v.x;
      w[2 * k + 1] = v.y;
    }
  }
  if (h) {
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] ^= upper_field_mask(k);
  }
  float2 v[NF / 2];
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int bit = 6 * i, wi = bit >> 5, o = bit & 31;
    // field i shifted to bit 7: table entry e of this lane is at e * 128 + lane * 4
    uint32_t f;
    if (o <= 26)
      f = o >= 7 ? (w[wi] >> (o - 7)) : (w[wi] << (7 - o));
    else
      f = __funnelshift_r(w[wi], w[wi + 1], o - 7);
    const float x = lds_f32_const(tab_lane + (f & (63u << 7)));
    if (i & 1)
      v[i >> 1].y = x;
    else
      v[i >> 1].x = x;
  }
  fwht_pairs<NF>(v);
  const float2 sc = make_float2(scale, scale);
#pragma unroll
  for (int g = 0; g < NF; g += 16) {
    float2 x[8];
    if (patched) {
      uint32_t acc[16];
      tmem_ld16(taddr + (uint32_t)(c_out + g), acc);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 8; ++e)
        x[e] = fma_f2(v[g / 2 + e], sc, make_float2(__uint_as_float(acc[2 * e]), __uint_as_float(acc[2 * e + 1])));
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = mul_f2(v[g / 2 + e], sc);
    }
    const uint4 o0 = make_uint4(pack2(x[0].x, x[0].y), pack2(x[1].x, x[1].y), pack2(x[2].x, x[2].y),
                                pack2(x[3].x, x[3].y));
    const uint4 o1 = make_uint4(pack2(x[4].x, x[4].y), pack2(x[5].x, x[5].y), pack2(x[6].x, x[6].y),
                                pack2(x[7].x, x[7].y));
    put16(rv.chunk(c_out + g), rv.chunk(c_out + g + 8), o0, o1, gdst, c_out + g);
  }
}

// ---- canonical-tile copies -----------------------------------------------------------------------

// Where the canonical rows of one row block come from: the store (or code)
// row of tile row 0, the bytes the loads of one tile deliver, the channel,
// and, in place, the pool row of each page segment (-1 = none).  The scalars
// stay apart from the segment array so that they live in registers.
struct SrcRB {
  int32_t src_row;
  uint32_t bytes;
  int32_t ch;
};

template <bool kComp>
__device__ __forceinline__ SrcRB rb_source(const Params& p, Walker& w, int64_t rb, int nbox, int nseg,
                                           int32_t (&seg_y)[BM / 8]) {
  walk_to(p, w, rb);
  const Tile t = decode(p, w, rb);
  SrcRB c;
  c.ch = t.ch;
  c.bytes = (uint32_t)nbox * BOX_BYTES;
  if (p.src_pool && !kComp) {
    c.bytes = 0;
    for (int sg = 0; sg < nseg; ++sg) {
      seg_y[sg] = segment(p, w, t, sg).y;
      if (seg_y[sg] >= 0) c.bytes += (uint32_t)nbox * (uint32_t)p.seg_rows * 128u;
    }
  }
  const int64_t t0 = t.pos0 - w.dst_pos;  // chunk token of tile row 0 (may be < 0)
  c.src_row = 0;
  if (kComp) {
    c.src_row = (int32_t)(p.comp_row_offset[w.chunk] + (int64_t)t.layer * w.T + t0);
    c.bytes = t.ch == 0 ? (uint32_t)p.BN * (uint32_t)BM : (uint32_t)(3 * p.BN / 8) * (uint32_t)BM;
  } else if (!p.src_pool) {
    c.src_row = (int32_t)(p.store_off[w.chunk] / p.D + ((int64_t)t.layer * p.n_ch_layout + t.ch) * w.T + t0);
  }
  return c;
}

// The TMA loads of column block cbi of a row block into stage st.
template <bool kComp>
__device__ __forceinline__ void tile_copy(const Params& p, const SrcRB c, const int32_t (&seg_y)[BM / 8], int cbi,
                                          int nbox, int nseg, uint8_t* st, uint64_t* bar) {
  const int col0 = (p.cb_first + cbi) * p.BN;
  if (kComp) {
    if (c.ch == 0) {
      for (int b = 0; b < p.BN / 128; ++b)
        tma_load_2d(st + p.out_bytes + b * BOX_BYTES, &p.kc_map, bar, col0 + b * 128, c.src_row);
    } else {
      tma_load_2d(st + p.out_bytes, &p.vc_map, bar, (p.cb_first + cbi) * (3 * p.BN / 8), c.src_row);
    }
  } else if (!p.src_pool) {
    for (int b = 0; b < nbox; ++b)
      tma_load_2d(st + b * BOX_BYTES, &p.src_map, bar, col0 + b * BOX_COLS, c.src_row);
  } else {
    for (int sg = 0; sg < nseg; ++sg) {
      if (seg_y[sg] < 0) continue;
      for (int b = 0; b < nbox; ++b)
        tma_load_2d(st + b * BOX_BYTES + (uint32_t)sg * p.seg_rows * 128u, &p.pool_map[c.ch], bar,
                    col0 + b * BOX_COLS, seg_y[sg]);
    }
  }
}

// ---- the kernel ----------------------------------------------------------------------------------

template <bool kPatch, bool kComp>
__global__ void __launch_bounds__(NUM_THREADS, 1) reuse_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem sm = carve_smem(smem_raw, p);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- set-up -------------------------------------------------------------------------------
  // A dependent launch may start its prologue now; everything this kernel
  // reads or writes in global memory comes after griddepcontrol.wait below.
  grid_launch_dependents();
  grid_dependency_wait();
  if (warp == 0) {
    // total row-block count: lanes split the items; only CTA 0 reports item-level errors
    int64_t n = 0;
    int32_t err = 0;
    Walker w;
    for (int32_t i = lane; i < p.n_items; i += 32) n += item_tiles(p, i, w, err);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
      err |= __shfl_xor_sync(0xFFFFFFFFu, err, o);
    }
    if (lane == 0) {
      // the compressed variant deals whole row blocks only: its decode epilogue
      // is register-bound, and the tail split's loop state measurably slows it
      sm.misc->full_rb = kComp ? n : n / gridDim.x * gridDim.x;
      sm.misc->tail_tiles = (n - sm.misc->full_rb) * p.n_cb;
      if (blockIdx.x == 0 && err && p.err_flag) atomicOr(p.err_flag, err);
    }
  }
  __syncthreads();
  if ((int64_t)blockIdx.x >= sm.misc->full_rb + sm.misc->tail_tiles) return;  // no work for this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], EPI_WARPS + 1);
      mbar_init(&sm.computed[s], EPI_WARPS);
    }
    for (int u = 0; u < p.uv_slots; ++u) {
      mbar_init(&sm.uv_full[u], 1);
      mbar_init(&sm.uv_empty[u], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], EPI_WARPS);
    }
    mbar_init(sm.drain, 1);
    sm.misc->abort_flag = 0;
    sm.misc->wait_limit = p.wait_limit_ns;
    fence_mbar_init();
  }
  if (kPatch) {
    // K groups the MMA reads but TMA never writes (rank 8 pads K to 16) stay zero
    const int kg_load = p.rank / 8 / p.ksplit;  // K groups a chunk's TMA box writes
    for (int u = 0; u < p.uv_slots; ++u) {
      uint8_t* slot = sm.uv + (size_t)u * (p.u_bytes + p.v_bytes);
      const uint32_t u_pad = (uint32_t)(p.kg_alloc - kg_load) * BM * 16u;
      const uint32_t v_pad = (uint32_t)(p.kg_alloc - kg_load) * p.BN * 16u;
      uint8_t* upad = slot + (uint32_t)kg_load * BM * 16u;
      uint8_t* vpad = slot + p.u_bytes + (uint32_t)kg_load * p.BN * 16u;
      for (uint32_t i = threadIdx.x * 16u; i < u_pad; i += NUM_THREADS * 16u)
        *reinterpret_cast<uint4*>(upad + i) = make_uint4(0, 0, 0, 0);
      for (uint32_t i = threadIdx.x * 16u; i < v_pad; i += NUM_THREADS * 16u)
        *reinterpret_cast<uint4*>(vpad + i) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    if (warp == 1) {
      tmem_alloc(&sm.misc->tmem_base, p.tmem_cols);
      tmem_relinquish();
    }
  }
  if (kComp)  // one copy of the centroid-sum table per lane: lane l reads only bank l
    for (int i = threadIdx.x; i < 64 * 32; i += NUM_THREADS) sm.table[i] = p.pair_sum[i >> 5];
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const int64_t full_rb = sm.misc->full_rb, n_units = kComp ? full_rb : full_rb + sm.misc->tail_tiles;
  const uint32_t tmem_base = kPatch ? sm.misc->tmem_base : 0u;
  const int nbox = p.BN / BOX_COLS;
  const int nseg = BM / p.seg_rows;
  const uint32_t uv_bytes = p.u_bytes + p.v_bytes;

  if (warp == 0) {
    // ================= TMA producer: canonical tiles =================
    if (lane == 0) {
      if (kComp) {
        tma_prefetch_desc(&p.kc_map);
        tma_prefetch_desc(&p.vc_map);
      } else {
        tma_prefetch_desc(p.src_pool ? &p.pool_map[0] : &p.src_map);
      }
      Walker w;
      walker_init(w);
      uint32_t it = 0;  // tiles loaded (stage fills)
      const uint32_t unarm_it = p.test_unarm ? 0u : 0xFFFFFFFFu;  // test only: the fill left unarmed
      bool go = true;
      for (int64_t u = blockIdx.x; go && u < n_units; u += gridDim.x) {
        const Unit un = kComp ? Unit{u, 0, p.n_cb} : unit_of(u, full_rb, p.n_cb);
        int32_t seg_y[BM / 8];
        const SrcRB c = rb_source<kComp>(p, w, un.rb, nbox, nseg, seg_y);
        for (int cbi = un.cb0; cbi < un.cb1; ++cbi, ++it) {
          const int s = (int)(it % (uint32_t)p.stages);
          const uint32_t ph = (it / (uint32_t)p.stages) & 1u;
          if (!wait_bounded(&sm.empty[s], ph ^ 1u, sm.misc, p.err_flag)) { go = false; break; }
          if (it == unarm_it) continue;  // test only: this stage's barrier is never armed
          mbar_arrive_expect_tx(&sm.full[s], c.bytes);
          tile_copy<kComp>(p, c, seg_y, cbi, nbox, nseg, sm.stages + (size_t)s * p.stage_bytes, &sm.full[s]);
        }
      }
      // drain: every stage's last fill must have landed before the CTA exits
      const uint32_t S = (uint32_t)p.stages;
      for (uint32_t s = 0; s < S && s < it; ++s) {
        const uint32_t fills = (it - s + S - 1) / S;
        wait_bounded(&sm.full[s], (fills - 1) & 1u, sm.misc, p.err_flag, false);
      }
    }
  } else if (warp == UV_WARP) {
    // ================= TMA producer: patch factors =================
    if (kPatch && lane == 0) {
      tma_prefetch_desc(&p.u_map);
      tma_prefetch_desc(&p.v_map);
      Walker w;
      walker_init(w);
      uint32_t pu = 0;
      bool go = true;
      for (int64_t u = blockIdx.x; go && u < n_units; u += gridDim.x) {
        const Unit un = kComp ? Unit{u, 0, p.n_cb} : unit_of(u, full_rb, p.n_cb);
        walk_to(p, w, un.rb);
        if (w.patch < 0) continue;
        const Tile t = decode(p, w, un.rb);
        const int64_t prow = p.patch_off[w.patch] / p.rank +
                             ((int64_t)t.layer * p.n_ch_layout + t.ch) * (int64_t)(w.T + p.D);
        const int32_t u_row = (int32_t)(prow + (t.pos0 - w.dst_pos));
        const int kg_chunk = p.rank / 8 / p.ksplit;  // K groups per chunk
        for (int cbi = un.cb0; cbi < un.cb1 && go; ++cbi) {
          for (int kc = 0; kc < p.ksplit; ++kc, ++pu) {
            const int ui = (int)(pu % (uint32_t)p.uv_slots);
            const uint32_t ph = (pu / (uint32_t)p.uv_slots) & 1u;
            if (!wait_bounded(&sm.uv_empty[ui], ph ^ 1u, sm.misc, p.err_flag)) { go = false; break; }
            uint8_t* slot = sm.uv + (size_t)ui * uv_bytes;
            mbar_arrive_expect_tx(&sm.uv_full[ui], (uint32_t)(BM + p.BN) * (uint32_t)kg_chunk * 16u);
            const int32_t v_row = (int32_t)(prow + w.T + (int64_t)(p.cb_first + cbi) * p.BN);
            if (!kComp && p.uv_row_bytes) {  // whole chunk rows, one request per row
              tma_load_2d(slot, &p.u_map, &sm.uv_full[ui], kc * kg_chunk * 8, u_row);
              tma_load_2d(slot + p.u_bytes, &p.v_map, &sm.uv_full[ui], kc * kg_chunk * 8, v_row);
            } else {
              tma_load_3d(slot, &p.u_map, &sm.uv_full[ui], 0, u_row, kc * kg_chunk);
              tma_load_3d(slot + p.u_bytes, &p.v_map, &sm.uv_full[ui], 0, v_row, kc * kg_chunk);
            }
          }
        }
      }
      const uint32_t S = (uint32_t)p.uv_slots;
      for (uint32_t u = 0; u < S && u < pu; ++u) {
        const uint32_t fills = (pu - u + S - 1) / S;
        wait_bounded(&sm.uv_full[u], (fills - 1) & 1u, sm.misc, p.err_flag, false);
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (kPatch && lane == 0) {
      const uint32_t idesc = umma_idesc_bf16_f32(BM, (uint32_t)p.BN);
      const uint32_t lbo_u = BM * 16u, lbo_v = (uint32_t)p.BN * 16u;
      const bool sw = !kComp && p.uv_row_bytes != 0;
      const uint32_t ainc = sw ? 2u : (2u * lbo_u) >> 4, binc = sw ? 2u : (2u * lbo_v) >> 4;
      Walker w;
      walker_init(w);
      uint32_t pt = 0, pc = 0;  // patched tiles, patch-factor chunks
      bool issued = false, go = true;
      for (int64_t u = blockIdx.x; go && u < n_units; u += gridDim.x) {
        const Unit un = kComp ? Unit{u, 0, p.n_cb} : unit_of(u, full_rb, p.n_cb);
        walk_to(p, w, un.rb);
        if (w.patch < 0) continue;
        for (int cbi = un.cb0; cbi < un.cb1 && go; ++cbi, ++pt) {
          const uint32_t buf = pt & 1u, tph = (pt >> 1) & 1u;
          if (!wait_bounded(&sm.tempty[buf], tph ^ 1u, sm.misc, p.err_flag)) { go = false; break; }
          for (int kc = 0; kc < p.ksplit; ++kc, ++pc) {
            const int ui = (int)(pc % (uint32_t)p.uv_slots);
            const uint32_t uph = (pc / (uint32_t)p.uv_slots) & 1u;
            if (!wait_bounded(&sm.uv_full[ui], uph, sm.misc, p.err_flag)) { go = false; break; }
            tc_fence_after_sync();
            const uint32_t ua = smem_addr(sm.uv + (size_t)ui * uv_bytes), va = ua + p.u_bytes;
            // descriptors of K step 0; step k starts k x (32 bytes into the swizzled rows, or two
            // core-matrix K groups) further, i.e. k x ainc / binc in the start-address field
            const uint64_t ad0 = sw ? umma_desc_kmajor_sw(ua, (uint32_t)p.uv_row_bytes)
                                    : umma_desc_kmajor_noswizzle(ua, lbo_u, 128u);
            const uint64_t bd0 = sw ? umma_desc_kmajor_sw(va, (uint32_t)p.uv_row_bytes)
                                    : umma_desc_kmajor_noswizzle(va, lbo_v, 128u);
            for (int k = 0; k < p.ksteps; ++k)
              umma_bf16(tmem_base + buf * (uint32_t)p.BN, ad0 + (uint64_t)(k * ainc), bd0 + (uint64_t)(k * binc),
                        idesc, (kc > 0 || k > 0) ? 1u : 0u);
            umma_commit(&sm.uv_empty[ui]);
            issued = true;
          }
          if (!go) break;
          umma_commit(&sm.tfull[buf]);
        }
      }
      if (issued) {
        umma_commit(sm.drain);
        wait_bounded(sm.drain, 0, sm.misc, p.err_flag, false);
      }
    }
  } else if (warp == 2) {
    // ================= TMA store issuer =================
    if (lane == 0) {
      Walker w;
      walker_init(w);
      uint32_t it = 0;
      bool go = true;
      for (int64_t u = blockIdx.x; go && u < n_units; u += gridDim.x) {
        const Unit un = kComp ? Unit{u, 0, p.n_cb} : unit_of(u, full_rb, p.n_cb);
        walk_to(p, w, un.rb);
        const Tile t = decode(p, w, un.rb);
        int32_t seg_y[BM / 8];  // pool row of each valid page segment, else -1
        bool seg_full[BM / 8];
        int lo8 = 0, hi8 = 0;   // 8-row sub-blocks of the row block inside the item: [lo8, hi8)
        {
          const int64_t a = w.dst_pos - t.pos0, b = w.dst_pos + w.T - t.pos0;
          lo8 = a <= 0 ? 0 : (int)((a + 7) >> 3);
          hi8 = b >= BM ? BM / 8 : (int)(b >> 3);
        }
        for (int sg = 0; sg < nseg; ++sg) {
          const Segment seg = segment(p, w, t, sg);
          seg_y[sg] = seg.y;
          seg_full[sg] = seg.full;
        }
        for (int cbi = un.cb0; cbi < un.cb1; ++cbi, ++it) {
          const int s = (int)(it % (uint32_t)p.stages);
          const uint32_t ph = (it / (uint32_t)p.stages) & 1u;
          if (!wait_bounded(&sm.computed[s], ph, sm.misc, p.err_flag)) { go = false; break; }
          // after a wait gave up, tiles may be marked computed without being so: store nothing more
          if (*reinterpret_cast<volatile int32_t*>(&sm.misc->abort_flag)) { go = false; break; }
          const uint8_t* st = sm.stages + (size_t)s * p.stage_bytes;
          const int col0 = (p.cb_first + cbi) * p.BN;
          for (int sg = 0; sg < nseg; ++sg) {
            if (seg_y[sg] < 0) continue;
            if (seg_full[sg]) {
              for (int b = 0; b < nbox; ++b)
                tma_store_2d(&p.pool_map[t.ch], st + b * BOX_BYTES + (uint32_t)sg * p.seg_rows * 128u,
                             col0 + b * BOX_COLS, seg_y[sg]);
              continue;
            }
            // partly covered page: its 8-row sub-blocks that lie inside the item
            const int r0 = sg * p.seg_rows;
            for (int k8 = r0 >> 3; k8 < ((r0 + p.seg_rows) >> 3); ++k8) {
              if (k8 < lo8 || k8 >= hi8) continue;
              for (int b = 0; b < nbox; ++b)
                tma_store_2d(&p.pool_map8[t.ch], st + b * BOX_BYTES + (uint32_t)k8 * 1024u, col0 + b * BOX_COLS,
                             seg_y[sg] + (k8 * 8 - r0));
            }
          }
          bulk_commit_group();
          bulk_wait_group_read0();  // the stage may be refilled once the stores have read it
          mbar_arrive(&sm.empty[s]);
        }
      }
      // the stages must outlive the stores' reads of them; the writes
      // themselves complete before the grid does
      bulk_wait_group_read0();
    }
  } else {
    // ================= epilogue (warps 3..10) =================
    const int e = warp - EPI_WARP0;      // 0..7
    const int h = e >> 2;                // column half
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int r = q * 32 + lane;         // tile row owned by this thread
    const int et = threadIdx.x - EPI_WARP0 * 32;  // 0..255
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    Walker w;
    walker_init(w);
    int32_t table_item[2] = {-1, -1};  // item whose phases each table holds
    uint32_t it = 0, pt = 0, uix = 0;  // tiles, patched tiles, units of this CTA
    bool ok = true;  // warp-uniform: every wait of this warp so far succeeded
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x, ++uix) {
      const Unit un = kComp ? Unit{u, 0, p.n_cb} : unit_of(u, full_rb, p.n_cb);
      walk_to(p, w, un.rb);
      Tile t = decode(p, w, un.rb);
      const bool patched = kPatch && w.patch >= 0;
      const bool rot = p.rotate && t.ch == 0;
      // destination of row r: rows of whole page segments go out with the TMA
      // store; rows of partly covered pages are stored by their own threads
      int64_t dst = -1;
      {
        const int64_t pos = t.pos0 + r;
        if (pos >= w.dst_pos && pos < w.dst_pos + w.T) {
          const Segment seg = segment(p, w, t, r >> p.seg_shift);
          if (seg.y < 0) {
            if (h == 0 && p.err_flag) atomicOr(p.err_flag, KAMERA_EFLAG_PAGE_OOB);
          } else if (!seg.full) {
            // an 8-row sub-block wholly inside the item goes out by TMA too
            const int k8 = r >> 3;
            const bool block_in = t.pos0 + k8 * 8 >= w.dst_pos && t.pos0 + k8 * 8 + 8 <= w.dst_pos + w.T;
            if (!block_in) dst = (int64_t)seg.y + (r & (p.seg_rows - 1));
          }
        }
      }
      // compressed store: this row's store row and the K scale of (chunk, layer)
      int64_t crow = -1;
      float kscale = 0.0f;
      if (kComp) {
        const int64_t tok = t.pos0 + r - w.dst_pos;
        if (tok >= 0 && tok < w.T) crow = p.comp_row_offset[w.chunk] + (int64_t)t.layer * w.T + tok;
        if (t.ch == 0) kscale = p.k_scale[(int64_t)w.chunk * p.num_layers + t.layer];
      }
      // phase tables alternate by unit parity: their previous readers
      // finished before the last joint barrier
      float2* cs = sm.cs + (uix & 1u) * pairs_pad(p.n_pairs);
      if (h == 1 && rot && w.item != table_item[uix & 1u]) {
        float* csf = reinterpret_cast<float*>(cs);
        for (int i = et - 128; i < p.n_pairs; i += 128) {
          const float2 v = phase_cs(i < p.sec_end0 ? w.d0 : (i < p.sec_end1 ? w.d1 : w.d2), p.theta[i]);
          csf[4 * (i >> 1) + (i & 1)] = v.x;
          csf[4 * (i >> 1) + 2 + (i & 1)] = v.y;
        }
      }
      if (rot) table_item[uix & 1u] = w.item;
      if (!named_bar_and(1, EPI_THREADS, ok)) break;  // joint decision, and the table is ready

      for (int cbi = un.cb0; cbi < un.cb1; ++cbi, ++it) {
        t.cb = p.cb_first + cbi;
        const int s = (int)(it % (uint32_t)p.stages);
        const uint32_t ph = (it / (uint32_t)p.stages) & 1u;
        const uint32_t buf = pt & 1u;
        float nrm[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // compressed V: ||v|| of the tile's heads in this row
        if (kComp && t.ch == 1 && crow >= 0) {
          const int hpt = p.BN / p.head_dim, H = p.D / p.head_dim;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < hpt) nrm[j] = __ldg(p.v_norm + crow * H + t.cb * hpt + j);
        }
        bool wok = ok && wait_bounded(&sm.full[s], ph, sm.misc, p.err_flag);
        if (wok && patched) wok = wait_bounded(&sm.tfull[buf], (pt >> 1) & 1u, sm.misc, p.err_flag);
        ok = __all_sync(0xFFFFFFFFu, wok);

        // compute phase: this thread's row, its half of the units, in place
        if (ok) {
          const RowView rv{smem_addr(sm.stages + (size_t)s * p.stage_bytes) + (uint32_t)r * 128u, (uint32_t)r & 7u};
          const uint32_t taddr = tmem_base + lane_addr + buf * (uint32_t)p.BN;
          uint16_t* gdst = dst >= 0 ? p.pool[t.ch] + dst * p.D + (int64_t)t.cb * p.BN : nullptr;
          if (patched) tc_fence_after_sync();
          if (kComp && t.ch == 1) {
            const uint32_t stg = smem_addr(sm.stages + (size_t)s * p.stage_bytes) + p.out_bytes;
            const uint32_t tab = smem_addr(sm.table) + 4u * (uint32_t)lane;
            const int hd = p.head_dim, hpt = p.BN / hd;
            const uint32_t row_codes = stg + (uint32_t)r * (3u * p.BN / 8u);
#pragma unroll 1
            for (int j = 0; j < hpt; ++j) {
              const float n = j == 0 ? nrm[0] : (j == 1 ? nrm[1] : (j == 2 ? nrm[2] : nrm[3]));
              const uint32_t codes = row_codes + (uint32_t)(j * 3 * hd / 8);
              if (hd == 128)
                epi_vhalf<128>(rv, codes, n * (1.0f / 128), h, j * 128 + h * 64, taddr, tab, gdst, patched);
              else
                epi_vhalf<64>(rv, codes, n * (1.0f / 64), h, j * 64 + h * 32, taddr, tab, gdst, patched);
            }
          } else if (kComp) {
            const uint32_t stg = smem_addr(sm.stages + (size_t)s * p.stage_bytes) + p.out_bytes;
            const SrcK8 src{stg + (uint32_t)r * 128u, (uint32_t)r & 7u, kscale};
            if (patched && p.frame == KAMERA_PATCH_CANONICAL_FRAME)
              epi_row<true, true, true>(p, src, rv, t.cb, rot, h, taddr, cs, gdst);
            else if (patched)
              epi_row<true, false, true>(p, src, rv, t.cb, rot, h, taddr, cs, gdst);
            else
              epi_row<false, false, true>(p, src, rv, t.cb, rot, h, taddr, cs, gdst);
          } else {
            const SrcTile src{rv};
            if (patched && p.frame == KAMERA_PATCH_CANONICAL_FRAME)
              epi_row<true, true, false>(p, src, rv, t.cb, rot, h, taddr, cs, gdst);
            else if (patched)
              epi_row<true, false, false>(p, src, rv, t.cb, rot, h, taddr, cs, gdst);
            else
              epi_row<false, false, false>(p, src, rv, t.cb, rot, h, taddr, cs, gdst);
          }
        }
        if (patched) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.tempty[buf]);
          ++pt;
        }
        fence_proxy_async_smem();  // in-place results -> visible to the TMA store
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.computed[s]);
          mbar_arrive(&sm.empty[s]);
        }
      }
    }
  }

  // ---- tear-down ---------------------------------------------------------------------------
  tc_fence_before_sync();
  __syncthreads();
  if (kPatch && warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace kamera
