/*
 * kamera.h -- C ABI of the GB300 (sm_103a) Kamera KV-reuse library.
 *
 * The operation (source: "Kamera: Unified Position-Invariant Multimodal KV
 * Cache for Training-Free Reuse", gist.science technical summary, §2
 * "Methodology: the Kamera operator"):
 *
 *     KV^(B|A) = R(delta) . KV(B|empty) + U_m V_m^T
 *
 * A canonical, position-free chunk K/V (KV(B|empty)) is gathered from a chunk
 * store, its keys are re-rotated by the RoPE phase shift delta of the new
 * position (§2 "Relocation R(delta)": an exact algebraic operation, not a
 * forward pass), a rank-m conditioning patch U_m V_m^T is added (§2 "Patch
 * application"), and the rows are scattered into a paged KV pool through a
 * block table.  §2 "Unified architecture support": MHA/GQA relocate the full
 * keys and patch K and V; MLA relocates only the decoupled 64-dim k_rope,
 * reuses c_KV byte for byte and patches both channels.  §3 names three window
 * operations, all served here: reorder with one shared orbit patch and recall
 * with a fresh patch (kamera_reuse_batched), sliding-window survival with
 * R(delta) only (kamera_relocate, in place).
 *
 * Conventions for every entry point:
 *   - Ownership: the caller owns every buffer.  The library allocates no
 *     memory, host or device, on any call.  Between calls it keeps only a
 *     per-device cache of launch facts (SM count, shared-memory limit), the
 *     static scratch array of kamera_factor_patches_noalloc and the launch
 *     tuning set by kamera_set_launch_tuning.
 *   - Pointers marked "device" must be device (or managed) memory of the
 *     current device; "host" pointers are read during the call only.
 *   - Asynchrony: work is enqueued on `stream`; KAMERA_OK means "validated and
 *     launched".  A launch failure returns KAMERA_ERR_CUDA.  Data-dependent
 *     problems (an id or page out of range) never fault: the affected item or
 *     row is skipped and a bit is OR-ed into *err_flag (device int32, may be
 *     NULL), readable after the caller synchronises the stream.  The caller
 *     clears *err_flag.
 *   - Layout: bf16 everywhere except the compressed store (int8 / 3-bit codes,
 *     see kamera_compressed_store).  D is the row width: num_kv_heads*head_dim for
 *     MHA/GQA, latent_dim + rope_dim for MLA.  Chunk store, per chunk c at
 *     element offset offset[c]: [layer][channel][len[c]][D] (channel 0 = K,
 *     1 = V; MLA has only channel 0, the latent row).  Patch store, per patch
 *     p at element offset offset[p]: for each layer and channel, U [len[p]][m]
 *     then V [D][m] (row-major, so V is V_m with its rows along D).  Pool: K
 *     and V each [layer][num_pages][page_size][D]; MLA uses only `k`.
 *     Position pos of sequence s lives at page block_table[s][pos/page_size],
 *     slot pos % page_size.
 *   - Alignment: every base pointer 16-byte aligned; D a multiple of 64;
 *     chunk offsets multiples of D; patch offsets multiples of m.
 *   - Aliasing: the source rows and the destination slots of one call must
 *     not overlap, except for the in-place modes, where each slot is read and
 *     written by the same item.  Two items writing the same slot is a caller
 *     error (the result is one of the two).
 *   - Launch shape: the reuse entry points pick the widest tile and the
 *     deepest pipeline that fit; kamera_set_launch_tuning (below) overrides
 *     that process-wide for tuning sweeps and tests.  Results do not depend
 *     on the launch shape.
 */
#ifndef KAMERA_H_
#define KAMERA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA stream type (cudaStream_t), declared without the CUDA headers. */
typedef struct CUstream_st* kamera_stream_t;

#define KAMERA_ABI_VERSION 4

typedef enum {
  KAMERA_OK = 0,
  KAMERA_ERR_NULL = 1,          /* a required pointer is NULL */
  KAMERA_ERR_INVALID_ARG = 2,   /* a size, count or enum is out of range */
  KAMERA_ERR_UNSUPPORTED = 3,   /* valid but not served (e.g. D not a multiple of 64) */
  KAMERA_ERR_ALIGNMENT = 4,     /* a base pointer is not 16-byte aligned */
  KAMERA_ERR_CUDA = 5           /* a CUDA call failed; see kamera_last_error() */
} kamera_status;

typedef enum { KAMERA_MHA = 0, KAMERA_GQA = 1, KAMERA_MLA = 2 } kamera_family;

/* RoPE pair convention: rotate-half pairs (i, i + d_r/2); interleaved (2i, 2i+1). */
typedef enum { KAMERA_ROTATE_HALF = 0, KAMERA_INTERLEAVED = 1 } kamera_pairing;

/* Where the patch is added: after the rotation (the literal equation
 * R(delta)KV + UV^T) or in the canonical frame, R(delta)(KV + UV^T). */
typedef enum { KAMERA_PATCH_AFTER_ROTATION = 0, KAMERA_PATCH_CANONICAL_FRAME = 1 } kamera_patch_frame;

/* Bits OR-ed into *err_flag by the kernels.  The offending item (or row, for
 * PAGE_OOB) is skipped; nothing traps. */
#define KAMERA_EFLAG_CHUNK_OOB 1  /* chunk id out of range, or its offset misaligned / past the store */
#define KAMERA_EFLAG_PAGE_OOB 2   /* sequence, block-table index or page id out of range */
#define KAMERA_EFLAG_PATCH_OOB 4  /* patch id out of range, or its offset misaligned / past the store */
#define KAMERA_EFLAG_LEN 8        /* n_tokens < 0, dst_pos < 0, or n_tokens != the chunk's / patch's length */
#define KAMERA_EFLAG_TIMEOUT 16   /* an internal pipeline wait gave up; the call's output is incomplete */

/* Model description (host struct, read during the call). */
typedef struct {
  int32_t family;         /* kamera_family */
  int32_t num_layers;     /* >= 1 */
  int32_t num_kv_heads;   /* MHA/GQA: >= 1 */
  int32_t head_dim;       /* MHA/GQA: 64, 128, 192 or 256 */
  int32_t rope_dim;       /* MHA/GQA: rotated dims per head, 0 = head_dim, a multiple of 64;
                             MLA: k_rope width (64) */
  int32_t latent_dim;     /* MLA: c_KV width (512), a multiple of 64 */
  int32_t pairing;        /* kamera_pairing */
  int32_t patch_frame;    /* kamera_patch_frame */
  double rope_base;       /* theta_i = rope_base^(-2i/rope_dim) when inv_freq is NULL */
  const double* inv_freq; /* host, [rope_dim/2] explicit theta_i table, or NULL */
  /* Multimodal RoPE (M-RoPE): the rope pairs split into consecutive temporal /
   * height / width sections, each turned by its own position component.
   * rope_sections = pairs per section, summing to rope_dim/2; all 0 = one
   * section (plain RoPE). */
  int32_t rope_sections[3];
  int32_t reserved0;            /* 0 */
  const int64_t* section_delta; /* device [n_items][3], per call: each item's shift of each section;
                                   NULL = every section takes the item's delta */
} kamera_model_desc;

/* Canonical chunk store: KV(B|empty) of every chunk (device memory). */
typedef struct {
  const void* data;       /* device bf16 [n_elems] */
  int64_t n_elems;        /* elements in data */
  const int64_t* offset;  /* device [n_chunks]: element offset of chunk c (a multiple of D) */
  const int32_t* len;     /* device [n_chunks]: tokens of chunk c */
  int32_t n_chunks;
} kamera_chunk_store;

/* Patch store: the rank-m conditioning patches U_m V_m^T (device memory). */
typedef struct {
  const void* data;       /* device bf16 [n_elems] */
  int64_t n_elems;
  const int64_t* offset;  /* device [n_patches]: element offset of patch p (a multiple of rank) */
  const int32_t* len;     /* device [n_patches]: tokens T_p the patch was formed for */
  int32_t n_patches;
  int32_t rank;           /* m: 8, 16, 32 or 64 (0 = no patches) */
} kamera_patch_store;

/* Paged KV pool and block table (device memory, written by the calls). */
typedef struct {
  void* k;                       /* device bf16 [num_layers][num_pages][page_size][D] */
  void* v;                       /* same shape; NULL for MLA */
  int64_t num_pages;
  int32_t page_size;             /* a power of two, >= 8 */
  const int32_t* block_table;    /* device int32 [n_seqs][max_pages_per_seq] */
  int32_t n_seqs;
  int32_t max_pages_per_seq;
} kamera_paged_pool;

/* One chunk reuse (device array of these; 32 bytes, naturally aligned). */
typedef struct {
  int32_t chunk_id;   /* index into the chunk store (ignored by the in-place calls) */
  int32_t patch_id;   /* index into the patch store; -1 = no patch for this item */
  int64_t delta;      /* RoPE phase shift in positions: new position - stored position */
  int32_t seq;        /* block-table row */
  int32_t n_tokens;   /* tokens; must equal the chunk's (and the patch's) length */
  int64_t dst_pos;    /* first logical position in the sequence */
} kamera_reuse_item;

/*
 * kamera_reuse_batched -- Kamera §2 reuse equation over a ragged batch.
 * For each item, layer, channel and token t: read the canonical row
 * (chunk_id, layer, channel, t), rotate the key row's RoPE pairs by
 * delta*theta_i (MLA: only the k_rope columns), add row t of U V^T of
 * (patch_id, layer, channel) if patch_id >= 0 and `patches` is not NULL, round
 * to bf16 (nearest even), and store it at position dst_pos + t of sequence
 * `seq`.  Serves reorder (§3, one orbit patch per chunk) and recall (§3, a
 * fresh patch).  `patches` NULL means no patch for any item.
 */
kamera_status kamera_reuse_batched(const kamera_model_desc* model, const kamera_chunk_store* store,
                                   const kamera_patch_store* patches, const kamera_reuse_item* items,
                                   int32_t n_items, const kamera_paged_pool* pool, int32_t* err_flag,
                                   kamera_stream_t stream);

/*
 * kamera_relocate -- Kamera §2 R(delta) alone.  With a chunk store it is
 * kamera_reuse_batched without patches.  With `store` NULL it works in place
 * on the pool (§3 sliding-window survival): the key rows at positions
 * dst_pos .. dst_pos+n_tokens-1 of each item are re-rotated by delta and
 * written back to the same slots; values (and MLA c_KV) are not touched.
 */
kamera_status kamera_relocate(const kamera_model_desc* model, const kamera_chunk_store* store,
                              const kamera_reuse_item* items, int32_t n_items, const kamera_paged_pool* pool,
                              int32_t* err_flag, kamera_stream_t stream);

/*
 * kamera_apply_patch -- Kamera §2 patch application alone, in place: for each
 * item with patch_id >= 0, add row t of U V^T of (patch_id, layer, channel) to
 * the pool row at position dst_pos + t, for K and V (MLA: the latent row), no
 * rotation.
 */
kamera_status kamera_apply_patch(const kamera_model_desc* model, const kamera_patch_store* patches,
                                 const kamera_reuse_item* items, int32_t n_items, const kamera_paged_pool* pool,
                                 int32_t* err_flag, kamera_stream_t stream);

/*
 * Patch formation -- Kamera §2 "Patch application": the patch is formed once
 * from the deficit Delta = KV(B|A) - KV(B|empty) by an SVD that keeps the top
 * m factors.  kamera_factor_patches computes, for every slab (one patch,
 * layer and channel), factors U_m [T][m] and V_m [D][m] whose product is the
 * rank-m truncation of Delta, and writes them as bf16 in the patch-store
 * layout (U of slab s at u_out + s*out_stride elements, V at v_out +
 * s*out_stride; for the slabs of one patch, u_out = patch base, v_out = patch
 * base + T*m, out_stride = (T+D)*m).  U_m has orthonormal columns; V_m carries
 * the singular values.
 *
 * Method: randomized range finder with q subspace iterations on a Gaussian
 * test matrix Omega [D][k], k = m + oversample (Halko, Martinsson & Tropp
 * 2011): the products with Delta on tensor cores with tf32 operands and fp32
 * accumulation (relative error per operand below 2^-10: when T, D, k and the
 * slab stride are multiples of 4 and Delta, Omega and the workspace 16-byte
 * aligned, Delta is read by TMA and truncated to tf32, otherwise rounded,
 * 2^-11; both below the bf16 rounding of the output factors), the
 * orthonormalisation and the small eigenproblem in fp32; exact (to that
 * rounding) when rank(Delta) <= k.  The caller passes
 * Omega, and scratch memory of kamera_factor_workspace_size() bytes.
 */
typedef struct {
  const float* delta;     /* device fp32: slab s at delta + s*delta_stride, [T][D] row-major */
  int64_t delta_stride;   /* elements between slabs (>= T*D) */
  int32_t n_slabs;
  int32_t T, D;           /* 1 <= T <= 8192, 1 <= D <= 2048 */
  int32_t rank;           /* m: 8, 16, 32 or 64 */
  int32_t oversample;     /* k = rank + oversample, 1 <= k <= 96 */
  int32_t power_iters;    /* q, 0..8 */
  const float* omega;     /* device fp32 [D][k] row-major */
} kamera_factor_desc;

/* Scratch bytes kamera_factor_patches needs for this description on the
 * current device (written to *bytes).  No allocation happens. */
kamera_status kamera_factor_workspace_size(const kamera_factor_desc* desc, size_t* bytes);

/* Form the factors (asynchronous on `stream`).  u_out / v_out: device bf16;
 * workspace: device, 256-byte aligned, at least the size above; its contents
 * are undefined afterwards. */
kamera_status kamera_factor_patches(const kamera_factor_desc* desc, void* u_out, void* v_out, int64_t out_stride,
                                    void* workspace, size_t workspace_bytes, kamera_stream_t stream);

/*
 * kamera_orbit_mean -- Kamera §3 "Reorder": one orbit patch, averaged over
 * permutations, serves every ordering of a cached set.  Given the deficits of
 * the same slabs measured under n sampled orderings (device fp32, ordering j
 * at deltas + j*ordering_stride, n_elems values each), write their mean
 *     out[e] = (sum_j deltas[j*ordering_stride + e]) / n
 * (fp32, the n terms added in index order, one correctly rounded division).
 * The mean is the deficit that kamera_factor_patches turns into the orbit
 * patch.  out may not overlap the inputs.  Asynchronous on `stream`.
 */
kamera_status kamera_orbit_mean(const float* deltas, int32_t n_orderings, int64_t ordering_stride, int64_t n_elems,
                                float* out, kamera_stream_t stream);

/*
 * kamera_factor_patches_noalloc -- the same patch formation for callers that
 * cannot allocate device memory.  No counterpart on the Kamera page: this is
 * a deployment convenience of this library.
 *
 * Who needs it: code whose device memory is owned entirely by another
 * allocator (a serving engine that carves its KV pool and buffers out of one
 * reservation), and plugin-style hooks whose enqueue step must neither
 * allocate nor risk the implicit device synchronisation that cudaMalloc and
 * cudaFree can cause.  Such callers cannot provide the workspace that
 * kamera_factor_patches asks for.
 *
 * The scratch instead lives in one static device array inside this library,
 * KAMERA_FACTOR_STATIC_SCRATCH_BYTES (16 MiB) per GPU, held by every GPU that
 * loads the library until the process exits.  The call allocates nothing and
 * never calls cudaMalloc / cudaFree.  Fewer CTAs may run than with a workspace
 * of full size (as many as the 16 MiB can serve), so it can be slower; the
 * results are the same.  A description whose single slab needs more scratch
 * than the array holds is rejected with KAMERA_ERR_UNSUPPORTED.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  The address is kept for the life of the process:
 * after cudaDeviceReset of a device the kept address is stale, so a process
 * that resets a device must not call this entry point on that device again.  All calls share the array and it keeps the last
 * call's contents; the kernel clears what it needs, so no caller action is
 * required -- but calls that overlap on the GPU (different streams, no
 * ordering between them) race on the array and must not be issued.
 */
#define KAMERA_FACTOR_STATIC_SCRATCH_BYTES (16u << 20)
kamera_status kamera_factor_patches_noalloc(const kamera_factor_desc* desc, void* u_out, void* v_out,
                                            int64_t out_stride, kamera_stream_t stream);

/*
 * Compressed canonical store -- the PolyKV scheme (source: "PolyKV: A Shared
 * Asymmetrically-Compressed KV Cache Pool for Multi-Agent LLM Inference",
 * gist.science summary, Spanish edition, §2B "asymmetric compression scheme
 * (TurboQuant MSE)"): keys as int8 with one linear scale per tensor; values at
 * 3 bits by rotating each vector with a fast Walsh-Hadamard transform so its
 * coordinates approach N(0,1), then mapping each coordinate to the nearest
 * Lloyd-Max centroid of N(0,1); decoding takes the centroid values and the
 * inverse transform.  Against bf16 the code bytes shrink 16 / ((8+3)/2) =
 * 2.91x (plus one fp32 norm per head row and one scale per (chunk, layer)).
 * MHA/GQA only, head_dim 64 or 128, D a multiple of 128.
 *
 * Layout (device memory).  Chunk c, layer l, token t is store row
 * row_offset[c] + l*len[c] + t.
 *   k_codes  int8  [n_rows][D]        code q of x: rint(x / s), in [-127, 127]
 *   k_scale  fp32  [n_chunks][layers] s = max|x| / 127 over that layer's K of
 *                                     the chunk (the "tensor"); decoded q * s
 *   v_codes  uint8 [n_rows][H][3*head_dim/8]: per head row of d = head_dim
 *                  values, 6-bit field i (i < d/2) = code[i] | code[i+d/2]<<3
 *                  at bit 6i (bit b of byte k is bit 8k+b)
 *   v_norm   fp32  [n_rows][H]        ||x|| of the head row
 * V codes: w = H x with H the Sylvester-ordered Hadamard matrix,
 * H[i][j] = (-1)^popcount(i&j); z = w / ||x||; code = the number of the seven
 * thresholds of kamera_v_codebook that are <= z (ascending centroids).
 * Decoded head row: (||x|| / d) * H c[code].
 */
typedef struct {
  void* k_codes;              /* device int8 [n_rows][D] */
  float* k_scale;             /* device fp32 [n_chunks][num_layers] */
  void* v_codes;              /* device uint8 [n_rows][num_kv_heads][3*head_dim/8] */
  float* v_norm;              /* device fp32 [n_rows][num_kv_heads] */
  const int64_t* row_offset;  /* device [n_chunks]: store row of (chunk c, layer 0, token 0) */
  const int32_t* len;         /* device [n_chunks]: tokens of chunk c */
  int32_t n_chunks;
  int32_t reserved;           /* 0 */
  int64_t n_rows;             /* rows of k_codes / v_codes / v_norm */
} kamera_compressed_store;

/*
 * kamera_v_codebook -- the V codebook (host call, no GPU): the 8 Lloyd-Max
 * centroids of N(0,1) rounded to fp32, ascending, exactly antisymmetric, and
 * the 7 thresholds (fp32 midpoints of neighbouring centroids).  Either pointer
 * may be NULL.
 */
kamera_status kamera_v_codebook(float centroids[8], float thresholds[7]);

/*
 * kamera_compress_chunks -- encode a bf16 chunk store (MHA/GQA layout
 * [layer][channel][len][D] per chunk) into `dst`: its k_codes, k_scale,
 * v_codes and v_norm are written; its row_offset, len, n_chunks and n_rows are
 * read (n_chunks must equal src->n_chunks; each chunk's len must match).
 * Every encoding decision is taken in fp32 in a fixed order (the transform's
 * butterflies with strides 1, 2, 4, ...; the sum of squares in index order
 * with fused multiply-add; IEEE division and square root), so the bytes are
 * reproducible.  A chunk whose lengths disagree or whose rows fall outside
 * either store is skipped with KAMERA_EFLAG_LEN / KAMERA_EFLAG_CHUNK_OOB.
 * dst may not overlap src.  Asynchronous on `stream`.
 */
kamera_status kamera_compress_chunks(const kamera_model_desc* model, const kamera_chunk_store* src,
                                     const kamera_compressed_store* dst, int32_t* err_flag, kamera_stream_t stream);

/*
 * kamera_reuse_compressed -- kamera_reuse_batched (Kamera §2 reuse equation)
 * whose canonical rows KV(B|empty) come from a compressed store: each row is
 * decoded (K: q * s; V: (||v|| / d) * H c[code]) in fp32 on the way from the
 * store to the tile, then rotated, patched, rounded to bf16 once and scattered
 * exactly as kamera_reuse_batched does.  Same items, pool, patches and error
 * bits (a chunk whose rows run past n_rows: KAMERA_EFLAG_CHUNK_OOB).
 */
kamera_status kamera_reuse_compressed(const kamera_model_desc* model, const kamera_compressed_store* store,
                                      const kamera_patch_store* patches, const kamera_reuse_item* items,
                                      int32_t n_items, const kamera_paged_pool* pool, int32_t* err_flag,
                                      kamera_stream_t stream);

/*
 * Launch tuning (no counterpart on the pages: a knob of this library).  One
 * process-wide setting, read by every later call of the reuse entry points
 * (kamera_reuse_batched, kamera_relocate, kamera_apply_patch,
 * kamera_reuse_compressed); a field left 0 keeps the library's own choice.
 * It exists for tuning sweeps and tests: the output bits do not depend on
 * bn, stages, uv_slots, ksplit, no_pdl or grid.  A shape that does not fit
 * a call (e.g. bn not dividing D) makes that call return
 * KAMERA_ERR_UNSUPPORTED.  Thread-safe; calls already enqueued keep the
 * setting they were launched with.
 */
typedef struct {
  int32_t bn;             /* tile width in columns: 64, 128, 192 or 256 */
  int32_t stages;         /* canonical tile stages in shared memory: 2..6 */
  int32_t uv_slots;       /* patch-factor slots: 1..8 */
  int32_t ksplit;         /* patch factors staged in 1, 2 or 4 parts of the rank */
  int32_t no_pdl;         /* non-zero: launch without programmatic dependent launch */
  int32_t grid;           /* CTAs of the persistent grid, 1..65535; 0 = one per SM */
  int64_t wait_limit_ns;  /* bound on every wait inside the kernel, 1 us .. 60 s; 0 = 2 s */
  /* TEST ONLY.  Non-zero: in every CTA the producer leaves the first canonical
   * stage unfilled and its barrier unarmed, so the waits on it run out after
   * wait_limit_ns.  The call then sets KAMERA_EFLAG_TIMEOUT, and each CTA
   * stops, waits (bounded) for its own copies and tensor-core work in flight,
   * releases its tensor memory and exits; the pool rows of the call are
   * incomplete.  This exercises the expiry path without any fault. */
  int32_t test_unarm_first_stage;
  int32_t reserved;       /* 0 */
} kamera_launch_tuning;

/* Set the process-wide tuning (NULL: back to the defaults, all fields 0).
 * KAMERA_ERR_INVALID_ARG for a field out of the ranges above. */
kamera_status kamera_set_launch_tuning(const kamera_launch_tuning* tuning);
/* Read the current setting. */
kamera_status kamera_get_launch_tuning(kamera_launch_tuning* tuning);

/* Human-readable name of a status code (static storage). */
const char* kamera_status_string(kamera_status status);

/* Detail of the last failed call on this thread ("" if none; thread-local storage). */
const char* kamera_last_error(void);

/* KAMERA_ABI_VERSION of the loaded library. */
int32_t kamera_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KAMERA_H_ */
