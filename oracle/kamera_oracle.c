/*
 * kamera_oracle.c -- plain, slow, fp64 CPU oracle of the Kamera KV-reuse operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) may link, load or call this file.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark use it.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes (source: "Kamera: Unified Position-Invariant Multimodal KV
 * Cache for Training-Free Reuse", gist.science technical summary, Italian and
 * Chinese editions -- cited below as "Kamera"):
 *
 *   Kamera §2 (Methodology, the Kamera operator), reuse equation:
 *       KV^(B|A) = R(delta) . KV(B|empty) + U_m V_m^T
 *   Kamera §2, "Relocation R(delta)": keys are re-rotated by the RoPE phase
 *       shift delta of the new position; an exact algebraic operation.
 *   Kamera §2, "Patch application": the rank-m patch U_m V_m^T is added.
 *   Kamera §2, "Unified architecture support": MHA/GQA relocate the full keys
 *       and patch K and V; MLA relocates only the decoupled 64-dim k_rope,
 *       reuses c_KV byte for byte and patches both channels.
 *   Kamera §3, the three window operations (reorder with an orbit patch,
 *       sliding-window survival with R(delta) only, recall with a fresh patch)
 *       are all instances of the same operator with different inputs.
 *   Kamera §2, patch formation: the top-m factors come from an SVD of the
 *       deficit; oracle_jacobi_svd below is a one-sided (Hestenes) Jacobi SVD
 *       used to build exact-rank test cases.
 *
 * Readings where the pages are silent (taken as follows):
 *   - RoPE pairs are rotate-half (i, i + d_r/2) unless interleaved (2i, 2i+1)
 *     is requested; theta_i = base^(-2i/d_r) unless a table is given.
 *   - delta is an integer position shift, the same for every token of a chunk.
 *     With multimodal RoPE (M-RoPE: the rope pairs split into consecutive
 *     temporal / height / width sections, each rotated by its own position
 *     component), each section has its own shift; one section = plain RoPE.
 *   - The patch is added after the rotation (the literal formula); the
 *     "canonical frame" variant rotates (KV + U V^T) instead.
 *   - Patch factors are per layer and per channel over the flattened H*d row
 *     (MLA: one U over the 576-wide latent row, V rows split 512 + 64).
 *   - Destination: position pos = dst_pos + t lands in page
 *     block_table[seq][pos / P], slot pos % P, of a pool laid out
 *     [layer][page][slot][D].
 *
 * Compressed canonical store (source: "PolyKV", gist.science summary, Spanish
 * edition, §2B "asymmetric compression scheme (TurboQuant MSE)"): K as int8
 * with one linear scale per tensor; V as 3-bit codes of the Walsh-Hadamard
 * rotated vector against the Lloyd-Max centroids of N(0,1), decoded by the
 * centroid values and the inverse transform.  The section "compressed
 * canonical store" below gives the encoder, the decoders and the reuse
 * operator reading such a store.
 *
 * Everything is evaluated in fp64 from the bf16 inputs (bf16 -> fp64 is exact).
 * Error bits follow the library's convention: an item whose chunk, patch,
 * length or sequence is invalid is skipped whole; a row whose page is invalid
 * is skipped alone.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_EFLAG_CHUNK_OOB 1
#define OR_EFLAG_PAGE_OOB 2
#define OR_EFLAG_PATCH_OOB 4
#define OR_EFLAG_LEN 8

enum { OR_MHA = 0, OR_GQA = 1, OR_MLA = 2 };
enum { OR_ROTATE_HALF = 0, OR_INTERLEAVED = 1 };
enum { OR_PATCH_AFTER_ROTATION = 0, OR_PATCH_CANONICAL_FRAME = 1 };
enum { OR_MODE_REUSE = 0, OR_MODE_RELOCATE_IN_PLACE = 1, OR_MODE_PATCH_IN_PLACE = 2 };

typedef struct {
  int32_t family;       /* OR_MHA, OR_GQA, OR_MLA */
  int32_t num_layers;
  int32_t num_kv_heads; /* MHA/GQA */
  int32_t head_dim;     /* MHA/GQA */
  int32_t rope_dim;     /* rotated dims per head (MHA/GQA, <= head_dim); MLA: k_rope width */
  int32_t latent_dim;   /* MLA: c_KV width (columns 0 .. latent_dim-1 of the latent row) */
  int32_t pairing;      /* OR_ROTATE_HALF or OR_INTERLEAVED */
  int32_t patch_frame;  /* OR_PATCH_AFTER_ROTATION or OR_PATCH_CANONICAL_FRAME */
  int32_t sections[3];  /* rope pairs per M-RoPE section (t, h, w); all 0 = a single section */
} oracle_model;

typedef struct {
  int32_t chunk_id;
  int32_t patch_id; /* -1: no patch */
  int64_t delta;
  int32_t seq;
  int32_t n_tokens;
  int64_t dst_pos;
} oracle_item;

/* ---- plain helpers --------------------------------------------------------- */

/* bf16 is the top half of an IEEE binary32; widening to fp64 is exact. */
static double bf16_bits_to_f64(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* Width of one K (or V) row: H*d for MHA/GQA, latent + k_rope for MLA. */
int32_t oracle_row_dim(const oracle_model* m) {
  if (m->family == OR_MLA) return m->latent_dim + m->rope_dim;
  return m->num_kv_heads * m->head_dim;
}

/* K and V are separate channels for MHA/GQA; MLA has one latent channel. */
int32_t oracle_num_channels(const oracle_model* m) { return m->family == OR_MLA ? 1 : 2; }

/* theta_i = base^(-2i/d_r), i < d_r/2 (the standard RoPE frequency ladder). */
void oracle_theta(double base, int32_t rope_dim, double* theta) {
  for (int32_t i = 0; i < rope_dim / 2; ++i) theta[i] = pow(base, -2.0 * (double)i / (double)rope_dim);
}

/*
 * R(delta) on one rotated region x[0 .. rope_dim-1]: every pair (a, b) turns
 * by the angle delta*theta_i,
 *     a' = a cos - b sin,   b' = b cos + a sin.
 * Kamera §2, "Relocation R(delta)".
 */
void oracle_rotate_region(double* x, int32_t rope_dim, const double* theta, int64_t delta, int32_t pairing) {
  int32_t half = rope_dim / 2;
  for (int32_t i = 0; i < half; ++i) {
    int32_t ia = (pairing == OR_INTERLEAVED) ? 2 * i : i;
    int32_t ib = (pairing == OR_INTERLEAVED) ? 2 * i + 1 : i + half;
    double phi = (double)delta * theta[i];
    double c = cos(phi), s = sin(phi);
    double a = x[ia], b = x[ib];
    x[ia] = a * c - b * s;
    x[ib] = b * c + a * s;
  }
}

/* R(delta) with one shift per M-RoPE section: pair i belongs to section s
 * when it lies in the s-th run of sections[s] consecutive pairs, and turns by
 * deltas[s]*theta_i.  With no sections every pair takes deltas[0]. */
void oracle_rotate_region_sections(double* x, int32_t rope_dim, const double* theta, const int64_t* deltas,
                                   const int32_t* sections, int32_t pairing) {
  int32_t half = rope_dim / 2;
  for (int32_t i = 0; i < half; ++i) {
    int32_t s = 0;
    if (sections[0] + sections[1] + sections[2] > 0) {
      if (i >= sections[0]) s = 1;
      if (i >= sections[0] + sections[1]) s = 2;
    }
    int32_t ia = (pairing == OR_INTERLEAVED) ? 2 * i : i;
    int32_t ib = (pairing == OR_INTERLEAVED) ? 2 * i + 1 : i + half;
    double phi = (double)deltas[s] * theta[i];
    double c = cos(phi), sn = sin(phi);
    double a = x[ia], b = x[ib];
    x[ia] = a * c - b * sn;
    x[ib] = b * c + a * sn;
  }
}

/* Apply R(delta) to every rotated region of a K row (channel 0).  The V row
 * (channel 1) carries no position and is never rotated.  MLA: only the k_rope
 * columns after the c_KV latent turn; c_KV is untouched.  deltas[0..2]: the
 * shift of each M-RoPE section (only deltas[0] without sections). */
void oracle_rotate_row(const oracle_model* m, const double* theta, int32_t channel, const int64_t* deltas,
                       double* row) {
  if (channel != 0) return;
  if (m->family == OR_MLA) {
    oracle_rotate_region_sections(row + m->latent_dim, m->rope_dim, theta, deltas, m->sections, m->pairing);
    return;
  }
  for (int32_t h = 0; h < m->num_kv_heads; ++h)
    oracle_rotate_region_sections(row + (int64_t)h * m->head_dim, m->rope_dim, theta, deltas, m->sections,
                                  m->pairing);
}

/* One output row of the operator, in fp64.
 *   src  [D]       canonical row (or pool row for the in-place modes)
 *   u    [rank]    this token's row of U, or NULL for no patch
 *   vmat [D][rank] V of this layer and channel
 * With the patch after rotation (the literal equation):  out = R src + U V^T row.
 * In the canonical frame:                                out = R (src + U V^T row). */
void oracle_row(const oracle_model* m, const double* theta, int32_t channel, const int64_t* deltas, int32_t rotate,
                const double* src, const double* u, const double* vmat, int32_t rank, double* out) {
  int32_t D = oracle_row_dim(m);
  double* patch = (double*)calloc((size_t)D, sizeof(double));
  if (u != NULL) {
    for (int32_t j = 0; j < D; ++j) {
      double acc = 0.0;
      for (int32_t r = 0; r < rank; ++r) acc += u[r] * vmat[(int64_t)j * rank + r];
      patch[j] = acc;
    }
  }
  if (m->patch_frame == OR_PATCH_CANONICAL_FRAME) {
    for (int32_t j = 0; j < D; ++j) out[j] = src[j] + patch[j];
    if (rotate) oracle_rotate_row(m, theta, channel, deltas, out);
  } else {
    for (int32_t j = 0; j < D; ++j) out[j] = src[j];
    if (rotate) oracle_rotate_row(m, theta, channel, deltas, out);
    for (int32_t j = 0; j < D; ++j) out[j] += patch[j];
  }
  free(patch);
}

/* Destination row (layer-independent part) of logical position pos of
 * sequence seq: page = block_table[seq][pos / P], slot = pos % P.
 * Returns page*P + slot, or -1 if the block-table index or the page id is out
 * of range. */
int64_t oracle_slot(const int32_t* block_table, int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                    int32_t seq, int64_t pos) {
  if (pos < 0) return -1;
  int64_t blk = pos / page_size;
  if (blk >= max_pages_per_seq) return -1;
  int64_t page = block_table[(int64_t)seq * max_pages_per_seq + blk];
  if (page < 0 || page >= num_pages) return -1;
  return page * page_size + pos % page_size;
}

/* ---- compressed canonical store ----------------------------------------------
 *
 * Source: "PolyKV" (gist.science summary, Spanish edition), §2B, the
 * asymmetric compression scheme (TurboQuant MSE):
 *   K: int8, linear quantisation with one scale per tensor.
 *   V: 3 bits per coordinate.  The vector is rotated by a fast Walsh-Hadamard
 *      transform, which spreads outliers and brings its coordinates close to
 *      N(0,1); each coordinate is mapped to the nearest precomputed Lloyd-Max
 *      centroid for N(0,1); decoding takes the centroid values and applies the
 *      inverse transform.
 *   Ratio against bf16: 16 / ((8 + 3) / 2) = 2.91.
 *
 * Readings (the page fixes none of these details):
 *   - A K "tensor" is one layer's K of one chunk, [T][D].  Scale
 *     s = max|x| / 127; code q = rint(x / s) clamped to [-127, 127] (s = 0:
 *     every code 0); decoded value q * s.
 *   - A V "vector" is one head's row of n = head_dim values (n a power of
 *     two).  H is the Sylvester-ordered Hadamard matrix, H[i][j] =
 *     (-1)^popcount(i & j), and w = H x.  The orthonormal rotation H/sqrt(n)
 *     gives coordinates of variance ||x||^2 / n, so the N(0,1)-normalised
 *     coordinate is z = w / ||x||.  Stored per head row: ||x|| (fp32) and
 *     the n codes.  Decoded value: (||x|| / n) * H c[code].
 *   - Codebook: the 8 Lloyd-Max centroids of N(0,1) rounded to fp32 (the
 *     upper four; the lower four are their exact negatives); thresholds: the
 *     fp32 midpoints of neighbouring centroids; code = the number of
 *     thresholds <= z (ascending centroid order, code 0 = most negative).
 *   - Packing: per head row 3n bits; 6-bit field i (i < n/2) holds
 *     code[i] | code[i + n/2] << 3 and starts at bit 6i of the row's bytes
 *     (bit b of byte k is bit 8k + b).
 *   - Store rows: chunk c, layer l, token t is row row_offset[c] + l*T + t of
 *     k_codes [rows][D], v_codes [rows][H][3n/8] and v_norm [rows][H];
 *     k_scale is [chunk][layer].  MHA/GQA only (MLA has no separate V).
 *   - The encoder's decisions are taken in fp32 with one fixed order of
 *     operations, which is part of the format: the in-place transform with
 *     strides 1, 2, 4, ...; the sum of squares in index order with fused
 *     multiply-add; IEEE division and square root.  The decoders are fp64.
 */

typedef struct {
  const int8_t* k_codes;      /* [n_rows][D] */
  const float* k_scale;       /* [n_chunks][num_layers] */
  const uint8_t* v_codes;     /* [n_rows][num_kv_heads][3*head_dim/8] */
  const float* v_norm;        /* [n_rows][num_kv_heads] */
  const int64_t* row_offset;  /* [n_chunks] */
  const int32_t* len;         /* [n_chunks] */
  int32_t n_chunks;
  int32_t reserved;
  int64_t n_rows;
  const float* codebook;      /* [8] fp32 centroids, ascending */
} oracle_cstore;

static double normal_pdf(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * acos(-1.0)); }
static double normal_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* Lloyd-Max quantiser of N(0,1) with `levels` levels (Lloyd 1957, Max 1960):
 * alternate the two optimality conditions,
 *     threshold k = midpoint of centroids k-1 and k,
 *     centroid k  = E[Z | t_k < Z < t_{k+1}] = (pdf(t_k) - pdf(t_{k+1})) / (cdf(t_{k+1}) - cdf(t_k)),
 * (t_0 = -inf, t_levels = +inf) starting from centroids spread evenly over
 * [-2, 2], until no centroid moves by more than 1e-15.  Returns the rounds used. */
int32_t oracle_lloyd_max_gaussian(int32_t levels, int32_t max_rounds, double* centroids) {
  double t[65];
  for (int32_t k = 0; k < levels; ++k) centroids[k] = -2.0 + 4.0 * (k + 0.5) / levels;
  int32_t round = 0;
  for (; round < max_rounds; ++round) {
    t[0] = -INFINITY;
    t[levels] = INFINITY;
    for (int32_t k = 1; k < levels; ++k) t[k] = 0.5 * (centroids[k - 1] + centroids[k]);
    double moved = 0.0;
    for (int32_t k = 0; k < levels; ++k) {
      double c = (normal_pdf(t[k]) - normal_pdf(t[k + 1])) / (normal_cdf(t[k + 1]) - normal_cdf(t[k]));
      moved = fmax(moved, fabs(c - centroids[k]));
      centroids[k] = c;
    }
    if (moved <= 1e-15) break;
  }
  return round;
}

/* The format's codebook: c32 [8] and thresholds t32 [7] (see the readings above). */
void oracle_v_codebook(float* c32, float* t32) {
  double c[8];
  oracle_lloyd_max_gaussian(8, 100000, c);
  for (int32_t k = 4; k < 8; ++k) {
    c32[k] = (float)c[k];
    c32[7 - k] = -c32[k];
  }
  for (int32_t k = 1; k < 8; ++k) t32[k - 1] = (c32[k - 1] + c32[k]) * 0.5f;
}

static float bf16_bits_to_f32(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return f;
}

/* K of one tensor of n bf16 values: the scale and the int8 codes (fp32 decisions). */
void oracle_quantize_k(const uint16_t* x, int64_t n, int8_t* q, float* scale) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(x[i])));
  const float s = amax / 127.0f;
  *scale = s;
  for (int64_t i = 0; i < n; ++i) {
    if (s == 0.0f) { q[i] = 0; continue; }
    float r = nearbyintf(bf16_bits_to_f32(x[i]) / s);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[i] = (int8_t)r;
  }
}

/* Code of element e of a packed head row of n codes. */
static int32_t v_code(const uint8_t* packed, int32_t n, int32_t e) {
  const int32_t half = n / 2;
  const int32_t bit0 = 6 * (e % half) + (e < half ? 0 : 3);
  int32_t code = 0;
  for (int32_t b = 0; b < 3; ++b) code |= ((packed[(bit0 + b) / 8] >> ((bit0 + b) % 8)) & 1) << b;
  return code;
}

/* V of one head row of n bf16 values (n <= 256): the packed codes (3n/8
 * bytes) and ||x||.  fp32 throughout, in the format's order of operations. */
void oracle_encode_v(const uint16_t* x_bits, int32_t n, const float* t32, uint8_t* packed, float* norm) {
  float x[256], w[256];
  if (n < 2 || n > 256) return;
  for (int32_t i = 0; i < n; ++i) w[i] = x[i] = bf16_bits_to_f32(x_bits[i]);
  for (int32_t h = 1; h < n; h *= 2)
    for (int32_t i = 0; i < n; i += 2 * h)
      for (int32_t j = i; j < i + h; ++j) {
        const float a = w[j], b = w[j + h];
        w[j] = a + b;
        w[j + h] = a - b;
      }
  float acc = 0.0f;
  for (int32_t i = 0; i < n; ++i) acc = fmaf(x[i], x[i], acc);
  const float nr = sqrtf(acc);
  *norm = nr;
  memset(packed, 0, (size_t)(3 * n / 8));
  for (int32_t e = 0; e < n; ++e) {
    int32_t code = 0;
    if (nr > 0.0f) {
      const float z = w[e] / nr;
      for (int32_t k = 0; k < 7; ++k) code += (t32[k] <= z) ? 1 : 0;
    }
    const int32_t bit0 = 6 * (e % (n / 2)) + (e < n / 2 ? 0 : 3);
    for (int32_t b = 0; b < 3; ++b) packed[(bit0 + b) / 8] |= (uint8_t)(((code >> b) & 1) << ((bit0 + b) % 8));
  }
}

/* Decoded head row: out[i] = (norm / n) * sum_j (-1)^popcount(i & j) * c32[code_j], in fp64. */
void oracle_decode_v(const uint8_t* packed, float norm, int32_t n, const float* c32, double* out) {
  for (int32_t i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int32_t j = 0; j < n; ++j) {
      const double c = (double)c32[v_code(packed, n, j)];
      acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -c : c;
    }
    out[i] = (double)norm / (double)n * acc;
  }
}

/* Canonical row (chunk c, layer l, channel ch, token t) of a compressed store, decoded in fp64. */
void oracle_decode_row(const oracle_model* m, const oracle_cstore* cs, int32_t c, int32_t l, int32_t ch, int32_t t,
                       double* out) {
  const int32_t D = oracle_row_dim(m);
  const int32_t H = m->num_kv_heads, n = m->head_dim;
  const int64_t row = cs->row_offset[c] + (int64_t)l * cs->len[c] + t;
  if (ch == 0) {
    const double s = (double)cs->k_scale[(int64_t)c * m->num_layers + l];
    for (int32_t j = 0; j < D; ++j) out[j] = (double)cs->k_codes[row * D + j] * s;
    return;
  }
  for (int32_t h = 0; h < H; ++h)
    oracle_decode_v(cs->v_codes + (row * H + h) * (3 * n / 8), cs->v_norm[row * H + h], n, cs->codebook,
                    out + (int64_t)h * n);
}

/* Encode a bf16 chunk store (per chunk [layer][channel][T][D], MHA/GQA) into
 * a compressed store whose row_offset / len the caller has set: one K scale
 * per (chunk, layer), every head row of V encoded on its own. */
void oracle_compress_store(const oracle_model* m, const uint16_t* store, const int64_t* store_off,
                           const int32_t* len, int32_t n_chunks, const int64_t* row_offset, const float* t32,
                           int8_t* k_codes, float* k_scale, uint8_t* v_codes, float* v_norm) {
  const int32_t D = oracle_row_dim(m);
  const int32_t H = m->num_kv_heads, n = m->head_dim, L = m->num_layers;
  for (int32_t c = 0; c < n_chunks; ++c) {
    const int64_t T = len[c];
    for (int32_t l = 0; l < L; ++l) {
      const uint16_t* k = store + store_off[c] + ((int64_t)l * 2 + 0) * T * D;
      const uint16_t* v = store + store_off[c] + ((int64_t)l * 2 + 1) * T * D;
      const int64_t row0 = row_offset[c] + (int64_t)l * T;
      oracle_quantize_k(k, T * D, k_codes + row0 * D, &k_scale[(int64_t)c * L + l]);
      for (int64_t t = 0; t < T; ++t)
        for (int32_t h = 0; h < H; ++h)
          oracle_encode_v(v + t * D + (int64_t)h * n, n, t32, v_codes + ((row0 + t) * H + h) * (3 * n / 8),
                          &v_norm[(row0 + t) * H + h]);
    }
  }
}

/*
 * The whole operator over a list of items, into fp64 images of the pool.
 *
 * mode OR_MODE_REUSE:             source rows come from the canonical chunk store
 *                                 (layout per chunk [layer][channel][T][D]); keys
 *                                 are rotated, the patch (if any) is added.
 * mode OR_MODE_RELOCATE_IN_PLACE: source rows are the pool's own K rows at the
 *                                 item's positions; only R(delta) applies, V is
 *                                 not touched (sliding-window survival, Kamera §3).
 * mode OR_MODE_PATCH_IN_PLACE:    source rows are the pool's rows; the patch is
 *                                 added to K and V with no rotation.
 *
 * Patch store layout per patch, per layer, per channel: U [T][rank] then
 * V [D][rank].  pool_*_in hold the pool's bf16 bits before the call; the fp64
 * images pool_*_out and the written masks are filled here (every slot starts
 * as its input value, unwritten).  pool_v_in / pool_v_out / wrote_v are
 * unused (may be NULL) for MLA.  section_deltas [n_items][3] gives each
 * item's per-section shifts when the model has M-RoPE sections (NULL: every
 * section takes the item's delta).  Returns the OR of the error bits.
 */
static int32_t reuse_impl(const oracle_model* m, const double* theta, int32_t mode,
                          const uint16_t* store, const int64_t* store_off, const int32_t* store_len, int32_t n_chunks,
                          const oracle_cstore* cs,
                          const uint16_t* patch, const int64_t* patch_off, const int32_t* patch_len,
                          int32_t n_patches, int32_t rank, const oracle_item* items, const int64_t* section_deltas,
                          int32_t n_items, const int32_t* block_table,
                          int32_t n_seqs, int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                          const uint16_t* pool_k_in, const uint16_t* pool_v_in, double* pool_k_out,
                          double* pool_v_out, uint8_t* wrote_k, uint8_t* wrote_v) {
  const int32_t D = oracle_row_dim(m);
  const int32_t L = m->num_layers;
  const int32_t n_ch = oracle_num_channels(m);
  const int64_t pool_rows = (int64_t)L * num_pages * page_size;
  int32_t err = 0;

  for (int64_t i = 0; i < pool_rows * D; ++i) {
    pool_k_out[i] = bf16_bits_to_f64(pool_k_in[i]);
    if (n_ch == 2) pool_v_out[i] = bf16_bits_to_f64(pool_v_in[i]);
  }
  memset(wrote_k, 0, (size_t)pool_rows);
  if (n_ch == 2) memset(wrote_v, 0, (size_t)pool_rows);

  double* src = (double*)malloc(sizeof(double) * (size_t)D);
  double* out = (double*)malloc(sizeof(double) * (size_t)D);
  double* u = (double*)malloc(sizeof(double) * (size_t)(rank > 0 ? rank : 1));
  double* vmat = (double*)malloc(sizeof(double) * (size_t)D * (size_t)(rank > 0 ? rank : 1));

  for (int32_t it = 0; it < n_items; ++it) {
    const oracle_item* item = &items[it];
    const int32_t T = item->n_tokens;
    if (T == 0) continue;
    if (T < 0 || item->dst_pos < 0) { err |= OR_EFLAG_LEN; continue; }
    if (item->seq < 0 || item->seq >= n_seqs) { err |= OR_EFLAG_PAGE_OOB; continue; }
    if (mode == OR_MODE_REUSE && cs == NULL) {
      if (item->chunk_id < 0 || item->chunk_id >= n_chunks) { err |= OR_EFLAG_CHUNK_OOB; continue; }
      if (store_len[item->chunk_id] != T) { err |= OR_EFLAG_LEN; continue; }
    }
    if (mode == OR_MODE_REUSE && cs != NULL) {
      if (item->chunk_id < 0 || item->chunk_id >= cs->n_chunks) { err |= OR_EFLAG_CHUNK_OOB; continue; }
      if (cs->len[item->chunk_id] != T) { err |= OR_EFLAG_LEN; continue; }
      const int64_t r0 = cs->row_offset[item->chunk_id];
      if (r0 < 0 || r0 + (int64_t)L * T > cs->n_rows) { err |= OR_EFLAG_CHUNK_OOB; continue; }
    }
    int32_t use_patch = 0;
    if (mode != OR_MODE_RELOCATE_IN_PLACE && rank > 0 && patch != NULL && item->patch_id >= 0) {
      if (item->patch_id >= n_patches) { err |= OR_EFLAG_PATCH_OOB; continue; }
      if (patch_len[item->patch_id] != T) { err |= OR_EFLAG_LEN; continue; }
      use_patch = 1;
    }
    if (mode == OR_MODE_PATCH_IN_PLACE && !use_patch) continue; /* nothing to add */
    const int32_t rotate = (mode != OR_MODE_PATCH_IN_PLACE);
    int64_t deltas[3] = {item->delta, item->delta, item->delta};
    if (section_deltas != NULL)
      for (int32_t s = 0; s < 3; ++s) deltas[s] = section_deltas[(int64_t)it * 3 + s];
    const int32_t ch_count = (mode == OR_MODE_RELOCATE_IN_PLACE) ? 1 : n_ch;

    for (int32_t l = 0; l < L; ++l) {
      for (int32_t ch = 0; ch < ch_count; ++ch) {
        const uint16_t* pin = (ch == 0) ? pool_k_in : pool_v_in;
        double* pout = (ch == 0) ? pool_k_out : pool_v_out;
        uint8_t* wrote = (ch == 0) ? wrote_k : wrote_v;
        if (use_patch) {
          const int64_t base = patch_off[item->patch_id] + ((int64_t)l * n_ch + ch) * (int64_t)(T + D) * rank;
          for (int64_t j = 0; j < D; ++j)
            for (int32_t r = 0; r < rank; ++r)
              vmat[j * rank + r] = bf16_bits_to_f64(patch[base + ((int64_t)T + j) * rank + r]);
        }
        for (int32_t t = 0; t < T; ++t) {
          const int64_t pos = item->dst_pos + t;
          const int64_t dst = oracle_slot(block_table, max_pages_per_seq, num_pages, page_size, item->seq, pos);
          if (dst < 0) { err |= OR_EFLAG_PAGE_OOB; continue; }
          const int64_t dst_row = (int64_t)l * num_pages * page_size + dst;
          if (mode == OR_MODE_REUSE && cs != NULL) {
            oracle_decode_row(m, cs, item->chunk_id, l, ch, t, src);
          } else if (mode == OR_MODE_REUSE) {
            const int64_t sb = store_off[item->chunk_id] + (((int64_t)l * n_ch + ch) * T + t) * D;
            for (int32_t j = 0; j < D; ++j) src[j] = bf16_bits_to_f64(store[sb + j]);
          } else {
            for (int32_t j = 0; j < D; ++j) src[j] = bf16_bits_to_f64(pin[dst_row * D + j]);
          }
          if (use_patch) {
            const int64_t ub = patch_off[item->patch_id] + ((int64_t)l * n_ch + ch) * (int64_t)(T + D) * rank +
                               (int64_t)t * rank;
            for (int32_t r = 0; r < rank; ++r) u[r] = bf16_bits_to_f64(patch[ub + r]);
          }
          oracle_row(m, theta, ch, deltas, rotate, src, use_patch ? u : NULL, vmat, rank, out);
          for (int32_t j = 0; j < D; ++j) pout[dst_row * D + j] = out[j];
          wrote[dst_row] = 1;
        }
      }
    }
  }
  free(src);
  free(out);
  free(u);
  free(vmat);
  return err;
}

int32_t oracle_reuse(const oracle_model* m, const double* theta, int32_t mode,
                     const uint16_t* store, const int64_t* store_off, const int32_t* store_len, int32_t n_chunks,
                     const uint16_t* patch, const int64_t* patch_off, const int32_t* patch_len, int32_t n_patches,
                     int32_t rank, const oracle_item* items, const int64_t* section_deltas, int32_t n_items,
                     const int32_t* block_table,
                     int32_t n_seqs, int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                     const uint16_t* pool_k_in, const uint16_t* pool_v_in, double* pool_k_out, double* pool_v_out,
                     uint8_t* wrote_k, uint8_t* wrote_v) {
  return reuse_impl(m, theta, mode, store, store_off, store_len, n_chunks, NULL, patch, patch_off, patch_len,
                    n_patches, rank, items, section_deltas, n_items, block_table, n_seqs, max_pages_per_seq,
                    num_pages, page_size, pool_k_in, pool_v_in, pool_k_out, pool_v_out, wrote_k, wrote_v);
}

/* The reuse operator (mode OR_MODE_REUSE) reading its canonical rows from a
 * compressed store: every source row is first decoded (oracle_decode_row),
 * then rotated, patched and scattered exactly as oracle_reuse does. */
int32_t oracle_reuse_compressed(const oracle_model* m, const double* theta, const oracle_cstore* cs,
                                const uint16_t* patch, const int64_t* patch_off, const int32_t* patch_len,
                                int32_t n_patches, int32_t rank, const oracle_item* items,
                                const int64_t* section_deltas, int32_t n_items, const int32_t* block_table,
                                int32_t n_seqs, int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                                const uint16_t* pool_k_in, const uint16_t* pool_v_in, double* pool_k_out,
                                double* pool_v_out, uint8_t* wrote_k, uint8_t* wrote_v) {
  return reuse_impl(m, theta, OR_MODE_REUSE, NULL, NULL, NULL, 0, cs, patch, patch_off, patch_len, n_patches, rank,
                    items, section_deltas, n_items, block_table, n_seqs, max_pages_per_seq, num_pages, page_size,
                    pool_k_in, pool_v_in, pool_k_out, pool_v_out, wrote_k, wrote_v);
}

/*
 * One-sided Jacobi SVD (Hestenes, 1958) of a rows x cols matrix a (row-major,
 * fp64), rows >= cols.  On return a holds U*Sigma (columns sorted by
 * decreasing norm), v [cols][cols] holds V (column j is the right singular
 * vector of singular value sigma[j]).  Each sweep orthogonalises every column
 * pair (p, q) by a plane rotation chosen so that the rotated pair is
 * orthogonal; it stops when every pair is orthogonal to the relative
 * tolerance.  Kamera §2 names the SVD as the step that extracts the top-m
 * patch factors; taking the first m columns gives U_m (with Sigma folded in)
 * and V_m.  Returns the number of sweeps used.
 */
int32_t oracle_jacobi_svd(double* a, int32_t rows, int32_t cols, double* v, double* sigma, int32_t max_sweeps) {
  for (int32_t i = 0; i < cols; ++i)
    for (int32_t j = 0; j < cols; ++j) v[(int64_t)i * cols + j] = (i == j) ? 1.0 : 0.0;
  int32_t sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
    int32_t rotated = 0;
    for (int32_t p = 0; p < cols - 1; ++p) {
      for (int32_t q = p + 1; q < cols; ++q) {
        double alpha = 0.0, beta = 0.0, gamma = 0.0;
        for (int32_t k = 0; k < rows; ++k) {
          double ap = a[(int64_t)k * cols + p], aq = a[(int64_t)k * cols + q];
          alpha += ap * ap;
          beta += aq * aq;
          gamma += ap * aq;
        }
        if (gamma == 0.0 || fabs(gamma) <= 1e-15 * sqrt(alpha * beta)) continue;
        rotated = 1;
        double zeta = (beta - alpha) / (2.0 * gamma);
        double t = (zeta >= 0.0 ? 1.0 : -1.0) / (fabs(zeta) + sqrt(1.0 + zeta * zeta));
        double c = 1.0 / sqrt(1.0 + t * t);
        double s = c * t;
        for (int32_t k = 0; k < rows; ++k) {
          double ap = a[(int64_t)k * cols + p], aq = a[(int64_t)k * cols + q];
          a[(int64_t)k * cols + p] = c * ap - s * aq;
          a[(int64_t)k * cols + q] = s * ap + c * aq;
        }
        for (int32_t k = 0; k < cols; ++k) {
          double vp = v[(int64_t)k * cols + p], vq = v[(int64_t)k * cols + q];
          v[(int64_t)k * cols + p] = c * vp - s * vq;
          v[(int64_t)k * cols + q] = s * vp + c * vq;
        }
      }
    }
    if (!rotated) break;
  }
  for (int32_t j = 0; j < cols; ++j) {
    double n2 = 0.0;
    for (int32_t k = 0; k < rows; ++k) n2 += a[(int64_t)k * cols + j] * a[(int64_t)k * cols + j];
    sigma[j] = sqrt(n2);
  }
  /* selection sort of the columns by decreasing sigma (cols is small) */
  for (int32_t j = 0; j < cols; ++j) {
    int32_t best = j;
    for (int32_t k = j + 1; k < cols; ++k)
      if (sigma[k] > sigma[best]) best = k;
    if (best == j) continue;
    double ts = sigma[j];
    sigma[j] = sigma[best];
    sigma[best] = ts;
    for (int32_t k = 0; k < rows; ++k) {
      double tmp = a[(int64_t)k * cols + j];
      a[(int64_t)k * cols + j] = a[(int64_t)k * cols + best];
      a[(int64_t)k * cols + best] = tmp;
    }
    for (int32_t k = 0; k < cols; ++k) {
      double tmp = v[(int64_t)k * cols + j];
      v[(int64_t)k * cols + j] = v[(int64_t)k * cols + best];
      v[(int64_t)k * cols + best] = tmp;
    }
  }
  return sweep;
}

/*
 * Orbit deficit (Kamera §3, "Reorder"): one orbit patch, averaged over
 * permutations, serves every ordering of a cached set.  The deficit it
 * factors is the mean of the deficits measured under n sampled orderings:
 *     out[e] = (1/n) * sum_j deltas[j*stride + e].
 */
void oracle_orbit_mean(const float* deltas, int32_t n, int64_t stride, int64_t n_elems, double* out) {
  for (int64_t e = 0; e < n_elems; ++e) {
    double s = 0.0;
    for (int32_t j = 0; j < n; ++j) s += (double)deltas[(int64_t)j * stride + e];
    out[e] = s / (double)n;
  }
}

/* ---- parity driver (tests only) ------------------------------------------------
 *
 * Checks a block of rows computed elsewhere (e.g. by the GPU) against the
 * operator's definition, row by row: for each row i of one (item, layer,
 * channel), the reference is oracle_row() of the canonical row src[i], the
 * patch row u[i] (NULL: no patch) and V (vmat, [D][rank]), and the row got[i]
 * (bf16 bits) must satisfy, element by element,
 *     |got - ref| <= ulp_bf16(ref) + abs_tol,
 *     ulp_bf16(x) = 2^(floor(log2(max(|x|, 2^-126))) - 7)
 * (one unit in the last place of bf16, which has 8 significant bits, plus an
 * absolute allowance near zero).  Columns [0, n_exact) must moreover equal
 * src bit for bit (MLA c_KV without a patch).  A NaN in got fails.
 * Returns the number of failing elements; *max_err is the largest |got - ref|
 * seen, *first_bad the index i*D + j of the first failure (or -1).  No state
 * outside its arguments, so callers may run blocks on several threads. */
/* The comparison of one row (D values) against its fp64 reference; updates
 * the failure count, the largest error and the first failing index (base = the
 * row's first element index).  exact: the canonical bits that columns
 * [0, n_exact) must equal, or NULL. */
static void compare_row(int32_t D, const double* ref, const uint16_t* got, const uint16_t* exact, int32_t n_exact,
                        double abs_tol, int64_t base, int64_t* bad, double* worst, int64_t* first_bad) {
  for (int32_t j = 0; j < D; ++j) {
    double g = bf16_bits_to_f64(got[j]);
    double err = fabs(g - ref[j]);
    int e2 = 0;
    double a = fabs(ref[j]);
    frexp(a > 0x1p-126 ? a : 0x1p-126, &e2); /* a = f * 2^e2, f in [0.5, 1): floor(log2 a) = e2 - 1 */
    double tol = ldexp(1.0, e2 - 1 - 7) + abs_tol;
    int ok = err <= tol; /* false for NaN */
    if (exact != NULL && j < n_exact && got[j] != exact[j]) ok = 0;
    if (err > *worst) *worst = err;
    if (!ok) {
      if (*first_bad < 0) *first_bad = base + j;
      ++*bad;
    }
  }
}

int64_t oracle_check_rows(const oracle_model* m, const double* theta, int32_t channel, const int64_t* deltas,
                          int32_t rotate, int32_t n_rows, const uint16_t* src, const uint16_t* u,
                          const uint16_t* vmat, int32_t rank, const uint16_t* got, int32_t n_exact, double abs_tol,
                          double* max_err, int64_t* first_bad) {
  int32_t D = oracle_row_dim(m);
  double* v = (double*)calloc((size_t)D * (size_t)(rank > 0 ? rank : 1), sizeof(double));
  double* s = (double*)malloc((size_t)D * sizeof(double));
  double* ur = (double*)malloc((size_t)(rank > 0 ? rank : 1) * sizeof(double));
  double* ref = (double*)malloc((size_t)D * sizeof(double));
  int64_t bad = 0;
  double worst = 0.0;
  *first_bad = -1;
  if (u != NULL)
    for (int64_t e = 0; e < (int64_t)D * rank; ++e) v[e] = bf16_bits_to_f64(vmat[e]);
  for (int32_t i = 0; i < n_rows; ++i) {
    const uint16_t* srow = src + (int64_t)i * D;
    for (int32_t j = 0; j < D; ++j) s[j] = bf16_bits_to_f64(srow[j]);
    if (u != NULL)
      for (int32_t r = 0; r < rank; ++r) ur[r] = bf16_bits_to_f64(u[(int64_t)i * rank + r]);
    oracle_row(m, theta, channel, deltas, rotate, s, u != NULL ? ur : NULL, v, rank, ref);
    compare_row(D, ref, got + (int64_t)i * D, srow, n_exact, abs_tol, (int64_t)i * D, &bad, &worst, first_bad);
  }
  free(v);
  free(s);
  free(ur);
  free(ref);
  *max_err = worst;
  return bad;
}

/* The same check for rows reused from a compressed store: the canonical row
 * of token t0 + i of (chunk, layer, channel) is decoded with oracle_decode_row
 * (real-valued, no bf16 rounding), then rotated, patched and compared as
 * above. */
int64_t oracle_check_rows_compressed(const oracle_model* m, const double* theta, const oracle_cstore* cs,
                                     int32_t chunk, int32_t layer, int32_t channel, int32_t t0,
                                     const int64_t* deltas, int32_t n_rows, const uint16_t* u, const uint16_t* vmat,
                                     int32_t rank, const uint16_t* got, double abs_tol, double* max_err,
                                     int64_t* first_bad) {
  int32_t D = oracle_row_dim(m);
  double* v = (double*)calloc((size_t)D * (size_t)(rank > 0 ? rank : 1), sizeof(double));
  double* s = (double*)malloc((size_t)D * sizeof(double));
  double* ur = (double*)malloc((size_t)(rank > 0 ? rank : 1) * sizeof(double));
  double* ref = (double*)malloc((size_t)D * sizeof(double));
  int64_t bad = 0;
  double worst = 0.0;
  *first_bad = -1;
  if (u != NULL)
    for (int64_t e = 0; e < (int64_t)D * rank; ++e) v[e] = bf16_bits_to_f64(vmat[e]);
  for (int32_t i = 0; i < n_rows; ++i) {
    oracle_decode_row(m, cs, chunk, layer, channel, t0 + i, s);
    if (u != NULL)
      for (int32_t r = 0; r < rank; ++r) ur[r] = bf16_bits_to_f64(u[(int64_t)i * rank + r]);
    oracle_row(m, theta, channel, deltas, 1, s, u != NULL ? ur : NULL, v, rank, ref);
    compare_row(D, ref, got + (int64_t)i * D, NULL, 0, abs_tol, (int64_t)i * D, &bad, &worst, first_bad);
  }
  free(v);
  free(s);
  free(ur);
  free(ref);
  *max_err = worst;
  return bad;
}
