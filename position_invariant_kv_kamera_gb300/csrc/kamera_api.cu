// kamera_api.cu -- host side of the C ABI declared in include/kamera.h:
// argument validation, the per-call work description (column blocks, RoPE
// pair table, theta ladder), TMA tensor maps, and the launch of the fused
// kernel.  No memory is allocated; the only per-call state is the kernel's
// parameter block.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "kamera.h"
#include "kamera_compress.cuh"
#include "kamera_factor_launch.h"
#include "kamera_orbit.cuh"
#include "kamera_kernel.cuh"

namespace kamera {
namespace {

thread_local std::string g_last_error;

kamera_status fail(kamera_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kamera_status fail(kamera_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

// ---- driver entry point for tensor-map encoding (no link-time libcuda dependency) ----
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

kamera_status encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                     const cuuint32_t* box, CUtensorMapSwizzle swz, const char* what,
                     CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(KAMERA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KAMERA_ERR_CUDA, "tensor map for %s: cuTensorMapEncodeTiled error %d", what, (int)r);
  return KAMERA_OK;
}

// ---- per-device launch facts ---------------------------------------------------------------
struct DeviceFacts {
  int sms = 0;
  int smem_optin = 0;
  bool attr_set[4] = {false, false, false, false};  // reuse kernel variants: shared-memory limit raised
  bool factor_attr_set = false;                     // both patch-formation instances
};
constexpr int kMaxDevices = 64;
DeviceFacts g_dev[kMaxDevices];
std::mutex g_dev_mu;

kamera_status device_facts(int* dev_out, DeviceFacts** facts) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(KAMERA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceFacts& f = g_dev[dev];
  if (f.sms == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(KAMERA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                  minor);
    cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&f.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  }
  *dev_out = dev;
  *facts = &f;
  return KAMERA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

// ---- the V codebook: Lloyd-Max quantiser of N(0,1), 8 levels ---------------------------------
// Symmetric form: the four positive centroids y_k with thresholds x_0 = 0,
// x_k = (y_{k-1} + y_k) / 2, x_4 = +inf; each y_k is the mean of N(0,1) over
// (x_k, x_{k+1}), (phi(x_k) - phi(x_{k+1})) / (Q(x_k) - Q(x_{k+1})) with Q the
// upper tail.  Iterated (Lloyd's method) from evenly spaced values until no
// centroid moves by more than 1e-16.
struct Codebook {
  float c[8];          // ascending, c[7-k] = -c[k]
  float t[7];          // (c[k] + c[k+1]) / 2 in fp32
  float pair_sum[64];  // c[a] + c[b] at a + 8b
};

const Codebook& codebook() {
  static Codebook cb;
  static std::once_flag once;
  std::call_once(once, [] {
    const double inv_sqrt2 = 0.70710678118654752440, inv_sqrt2pi = 0.39894228040143267794;
    auto phi = [&](double x) { return std::isinf(x) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * x * x); };
    auto tail = [&](double x) { return std::isinf(x) ? 0.0 : 0.5 * std::erfc(x * inv_sqrt2); };
    double y[4] = {0.25, 0.75, 1.25, 1.75}, x[5];
    for (int round = 0; round < 200000; ++round) {
      x[0] = 0.0;
      x[4] = INFINITY;
      for (int k = 1; k < 4; ++k) x[k] = 0.5 * (y[k - 1] + y[k]);
      double moved = 0.0;
      for (int k = 0; k < 4; ++k) {
        const double yk = (phi(x[k]) - phi(x[k + 1])) / (tail(x[k]) - tail(x[k + 1]));
        moved = std::fmax(moved, std::fabs(yk - y[k]));
        y[k] = yk;
      }
      if (moved <= 1e-16) break;
    }
    for (int k = 0; k < 4; ++k) {
      cb.c[4 + k] = (float)y[k];
      cb.c[3 - k] = -cb.c[4 + k];
    }
    for (int k = 0; k < 7; ++k) cb.t[k] = (cb.c[k] + cb.c[k + 1]) * 0.5f;
    for (int a = 0; a < 8; ++a)
      for (int b = 0; b < 8; ++b) cb.pair_sum[a + 8 * b] = cb.c[a] + cb.c[b];
  });
  return cb;
}

enum Mode { MODE_REUSE = 0, MODE_RELOCATE_IN_PLACE = 1, MODE_PATCH_IN_PLACE = 2 };

// Process-wide launch tuning (kamera_set_launch_tuning): copied under the lock
// at each call, so a call never sees a half-written setting.
kamera_launch_tuning g_tuning = {};
std::mutex g_tuning_mu;

kamera_launch_tuning current_tuning() {
  std::lock_guard<std::mutex> lk(g_tuning_mu);
  return g_tuning;
}

kamera_status set_tuning(const kamera_launch_tuning* t) {
  g_last_error.clear();
  kamera_launch_tuning v = {};
  if (t) {
    v = *t;
    if (v.bn != 0 && v.bn != 64 && v.bn != 128 && v.bn != 192 && v.bn != 256)
      return fail(KAMERA_ERR_INVALID_ARG, "tuning: bn = %d (0, 64, 128, 192 or 256)", v.bn);
    if (v.stages != 0 && (v.stages < 2 || v.stages > 6))
      return fail(KAMERA_ERR_INVALID_ARG, "tuning: stages = %d (0 or 2..6)", v.stages);
    if (v.uv_slots < 0 || v.uv_slots > 8) return fail(KAMERA_ERR_INVALID_ARG, "tuning: uv_slots = %d", v.uv_slots);
    if (v.ksplit != 0 && v.ksplit != 1 && v.ksplit != 2 && v.ksplit != 4)
      return fail(KAMERA_ERR_INVALID_ARG, "tuning: ksplit = %d (0, 1, 2 or 4)", v.ksplit);
    if (v.grid < 0 || v.grid > 65535) return fail(KAMERA_ERR_INVALID_ARG, "tuning: grid = %d", v.grid);
    if (v.wait_limit_ns != 0 && (v.wait_limit_ns < 1000 || v.wait_limit_ns > 60000000000ll))
      return fail(KAMERA_ERR_INVALID_ARG, "tuning: wait_limit_ns = %lld (0 or 1e3 .. 6e10)",
                  (long long)v.wait_limit_ns);
    if (v.reserved != 0) return fail(KAMERA_ERR_INVALID_ARG, "tuning: reserved must be 0");
  }
  std::lock_guard<std::mutex> lk(g_tuning_mu);
  g_tuning = v;
  return KAMERA_OK;
}

kamera_status launch(Mode mode, const kamera_model_desc* model, const kamera_chunk_store* store,
                     const kamera_patch_store* patches, const kamera_reuse_item* items, int32_t n_items,
                     const kamera_paged_pool* pool, int32_t* err_flag, kamera_stream_t stream,
                     const kamera_compressed_store* cstore = nullptr) {
  g_last_error.clear();
  const bool comp = cstore != nullptr;
  if (!model) return fail(KAMERA_ERR_NULL, "model is NULL");
  if (!pool) return fail(KAMERA_ERR_NULL, "pool is NULL");
  if (n_items < 0) return fail(KAMERA_ERR_INVALID_ARG, "n_items = %d", n_items);
  if (n_items > 0 && !items) return fail(KAMERA_ERR_NULL, "items is NULL");
  if (mode == MODE_REUSE && !store && !comp) return fail(KAMERA_ERR_NULL, "chunk store is NULL");
  if (mode == MODE_PATCH_IN_PLACE && !patches) return fail(KAMERA_ERR_NULL, "patch store is NULL");

  // ---- model -----------------------------------------------------------------------------
  const int fam = model->family;
  if (fam != KAMERA_MHA && fam != KAMERA_GQA && fam != KAMERA_MLA)
    return fail(KAMERA_ERR_INVALID_ARG, "family = %d", fam);
  if (model->num_layers < 1) return fail(KAMERA_ERR_INVALID_ARG, "num_layers = %d", model->num_layers);
  if (model->pairing != KAMERA_ROTATE_HALF && model->pairing != KAMERA_INTERLEAVED)
    return fail(KAMERA_ERR_INVALID_ARG, "pairing = %d", model->pairing);
  if (model->patch_frame != KAMERA_PATCH_AFTER_ROTATION && model->patch_frame != KAMERA_PATCH_CANONICAL_FRAME)
    return fail(KAMERA_ERR_INVALID_ARG, "patch_frame = %d", model->patch_frame);
  int D = 0, rope = 0, heads = 0, head_stride = 0, rope_col0 = 0, n_ch_layout = 2;
  if (fam == KAMERA_MLA) {
    if (model->latent_dim < 64 || model->latent_dim % 64 != 0)
      return fail(KAMERA_ERR_UNSUPPORTED, "MLA latent_dim = %d (a positive multiple of 64 is served)",
                  model->latent_dim);
    rope = model->rope_dim;
    if (rope < 64 || rope % 64 != 0) return fail(KAMERA_ERR_UNSUPPORTED, "MLA rope_dim = %d", rope);
    D = model->latent_dim + rope;
    heads = 1;
    head_stride = rope;
    rope_col0 = model->latent_dim;
    n_ch_layout = 1;
    if (pool->v) return fail(KAMERA_ERR_INVALID_ARG, "MLA pools hold latent rows in `k`; `v` must be NULL");
  } else {
    if (model->num_kv_heads < 1) return fail(KAMERA_ERR_INVALID_ARG, "num_kv_heads = %d", model->num_kv_heads);
    const int hd = model->head_dim;
    if (hd < 64 || hd > 256 || hd % 64 != 0)
      return fail(KAMERA_ERR_UNSUPPORTED, "head_dim = %d (64, 128, 192 or 256 are served)", hd);
    rope = model->rope_dim == 0 ? hd : model->rope_dim;
    if (rope < 64 || rope > hd || rope % 64 != 0)
      return fail(KAMERA_ERR_UNSUPPORTED, "rope_dim = %d (a multiple of 64 up to head_dim)", rope);
    D = model->num_kv_heads * hd;
    heads = model->num_kv_heads;
    head_stride = hd;
  }
  if (D > 32 * MAX_GROUPS) return fail(KAMERA_ERR_UNSUPPORTED, "row width D = %d exceeds %d", D, 32 * MAX_GROUPS);
  if (comp) {
    if (fam == KAMERA_MLA) return fail(KAMERA_ERR_UNSUPPORTED, "the compressed store holds separate K and V (MHA/GQA)");
    if (model->head_dim != 64 && model->head_dim != 128)
      return fail(KAMERA_ERR_UNSUPPORTED, "compressed store: head_dim = %d (64 or 128 served)", model->head_dim);
    if (D % 128 != 0) return fail(KAMERA_ERR_UNSUPPORTED, "compressed store: D = %d (a multiple of 128 served)", D);
  }
  const int n_pairs = rope / 2;
  if (n_pairs > MAX_PAIRS) return fail(KAMERA_ERR_UNSUPPORTED, "rope_dim = %d", rope);
  const int* sec = model->rope_sections;
  if (sec[0] < 0 || sec[1] < 0 || sec[2] < 0)
    return fail(KAMERA_ERR_INVALID_ARG, "rope_sections = {%d, %d, %d}", sec[0], sec[1], sec[2]);
  const int sec_sum = sec[0] + sec[1] + sec[2];
  if (sec_sum != 0 && sec_sum != n_pairs)
    return fail(KAMERA_ERR_INVALID_ARG, "rope_sections sum to %d, not rope_dim/2 = %d", sec_sum, n_pairs);
  if (model->section_delta && (reinterpret_cast<uintptr_t>(model->section_delta) & 7u))
    return fail(KAMERA_ERR_ALIGNMENT, "section_delta must be 8-byte aligned");

  // ---- pool --------------------------------------------------------------------------------
  if (!pool->k) return fail(KAMERA_ERR_NULL, "pool->k is NULL");
  const bool need_v = fam != KAMERA_MLA && mode != MODE_RELOCATE_IN_PLACE;
  if (need_v && !pool->v) return fail(KAMERA_ERR_NULL, "pool->v is NULL");
  if (!aligned16(pool->k) || (pool->v && !aligned16(pool->v)))
    return fail(KAMERA_ERR_ALIGNMENT, "pool base pointers must be 16-byte aligned");
  if (!pool->block_table) return fail(KAMERA_ERR_NULL, "pool->block_table is NULL");
  if (pool->num_pages < 1 || pool->n_seqs < 1 || pool->max_pages_per_seq < 1)
    return fail(KAMERA_ERR_INVALID_ARG, "pool: num_pages=%lld n_seqs=%d max_pages_per_seq=%d",
                (long long)pool->num_pages, pool->n_seqs, pool->max_pages_per_seq);
  if (!pow2(pool->page_size) || pool->page_size < 8 || pool->page_size > (1 << 20))
    return fail(KAMERA_ERR_INVALID_ARG, "page_size = %d (a power of two >= 8)", pool->page_size);
  const int64_t pool_rows = (int64_t)model->num_layers * pool->num_pages * pool->page_size;
  if (pool_rows >= (int64_t(1) << 31))
    return fail(KAMERA_ERR_UNSUPPORTED, "pool has %lld rows per channel (< 2^31 served)", (long long)pool_rows);
  if (err_flag && (reinterpret_cast<uintptr_t>(err_flag) & 3u))
    return fail(KAMERA_ERR_ALIGNMENT, "err_flag must be 4-byte aligned");

  // ---- stores --------------------------------------------------------------------------------
  if (comp) {
    if (!cstore->k_codes || !cstore->k_scale || !cstore->v_codes || !cstore->v_norm || !cstore->row_offset ||
        !cstore->len)
      return fail(KAMERA_ERR_NULL, "compressed store: a pointer is NULL");
    if (!aligned16(cstore->k_codes) || !aligned16(cstore->v_codes) ||
        (reinterpret_cast<uintptr_t>(cstore->k_scale) & 3u) || (reinterpret_cast<uintptr_t>(cstore->v_norm) & 3u) ||
        (reinterpret_cast<uintptr_t>(cstore->row_offset) & 7u) || (reinterpret_cast<uintptr_t>(cstore->len) & 3u))
      return fail(KAMERA_ERR_ALIGNMENT, "compressed store: codes 16-byte aligned, the other arrays naturally");
    if (cstore->n_chunks < 0 || cstore->n_rows < 0 || cstore->reserved != 0)
      return fail(KAMERA_ERR_INVALID_ARG, "compressed store: n_chunks = %d, n_rows = %lld", cstore->n_chunks,
                  (long long)cstore->n_rows);
    if (cstore->n_rows >= (int64_t(1) << 31))
      return fail(KAMERA_ERR_UNSUPPORTED, "compressed store has %lld rows (< 2^31 served)", (long long)cstore->n_rows);
  }
  const bool use_store = mode == MODE_REUSE && !comp;
  int64_t store_rows = 0;
  if (use_store) {
    if (!store->data || !store->offset || !store->len)
      return fail(KAMERA_ERR_NULL, "chunk store data/offset/len is NULL");
    if (!aligned16(store->data)) return fail(KAMERA_ERR_ALIGNMENT, "chunk store data must be 16-byte aligned");
    if (store->n_chunks < 0 || store->n_elems < 0) return fail(KAMERA_ERR_INVALID_ARG, "chunk store sizes");
    store_rows = store->n_elems / D;
    if (store_rows >= (int64_t(1) << 31))
      return fail(KAMERA_ERR_UNSUPPORTED, "chunk store has %lld rows (< 2^31 served)", (long long)store_rows);
  }
  const bool use_patch = mode != MODE_RELOCATE_IN_PLACE && patches && patches->rank > 0;
  int rank = 0;
  int64_t patch_rows = 0;
  if (use_patch) {
    rank = patches->rank;
    if (rank != 8 && rank != 16 && rank != 32 && rank != 64)
      return fail(KAMERA_ERR_INVALID_ARG, "rank = %d (8, 16, 32 or 64)", rank);
    if (!patches->data || !patches->offset || !patches->len)
      return fail(KAMERA_ERR_NULL, "patch store data/offset/len is NULL");
    if (!aligned16(patches->data)) return fail(KAMERA_ERR_ALIGNMENT, "patch store data must be 16-byte aligned");
    if (patches->n_patches < 0 || patches->n_elems < 0) return fail(KAMERA_ERR_INVALID_ARG, "patch store sizes");
    patch_rows = patches->n_elems / rank;
    if (patch_rows >= (int64_t(1) << 31))
      return fail(KAMERA_ERR_UNSUPPORTED, "patch store has %lld rows (< 2^31 served)", (long long)patch_rows);
  } else if (patches && patches->rank < 0) {
    return fail(KAMERA_ERR_INVALID_ARG, "rank = %d", patches->rank);
  }
  if (mode == MODE_PATCH_IN_PLACE && !use_patch) return KAMERA_OK;  // rank 0: nothing to add
  if (n_items == 0) return KAMERA_OK;

  // ---- theta ladder and the key row's group table --------------------------------------------
  Params p;
  memset(&p, 0, sizeof p);
  for (int i = 0; i < n_pairs; ++i) {
    if (model->inv_freq) {
      p.theta[i] = model->inv_freq[i];
    } else {
      if (!(model->rope_base > 0.0) || !std::isfinite(model->rope_base))
        return fail(KAMERA_ERR_INVALID_ARG, "rope_base = %g", model->rope_base);
      p.theta[i] = std::pow(model->rope_base, -2.0 * (double)i / (double)rope);
    }
    if (!std::isfinite(p.theta[i])) return fail(KAMERA_ERR_INVALID_ARG, "theta[%d] is not finite", i);
  }
  const int n_groups = D / 32;
  for (int h = 0; h < heads; ++h) {
    const int a = rope_col0 + h * head_stride;  // first rotated column of this region
    for (int c = 0; c < rope; c += 32) {
      const int g = (a + c) / 32;
      if (model->pairing == KAMERA_INTERLEAVED) {
        p.group_kind[g] = GK_INTERLEAVED;
        p.pair_base[g] = (uint8_t)(c / 2);
      } else if (c < rope / 2) {
        p.group_kind[g] = (int8_t)(rope / 2 / 32);
        p.pair_base[g] = (uint8_t)c;
      } else {
        p.group_kind[g] = GK_SECOND;
      }
    }
  }

  {
    // alternate whole rotation units (and plain groups) between the two epilogue halves
    int k = 0;
    for (int g = 0; g < n_groups; ++g) {
      if (p.group_kind[g] == GK_SECOND) continue;
      p.owner0[g] = (uint8_t)(k++ & 1);
    }
  }

  // ---- tile shape: BN columns per tile, smem stages ---------------------------------------------
  int dev = 0;
  DeviceFacts* facts = nullptr;
  if (kamera_status st = device_facts(&dev, &facts)) return st;
  const kamera_launch_tuning tune = current_tuning();
  const int bn_env = tune.bn, st_env = tune.stages, uv_env = tune.uv_slots, ks_env = tune.ksplit;
  int BN = 0, stages = 0, uv_slots = 0, ksplit = 1, kg_alloc = 0;
  uint32_t stage_bytes = 0, uv_slot_bytes = 0;
  // compressed: the stage also holds the codes (BN*128 bytes for K, more than
  // the 3BN/8 * 128 of V), plus the replicated centroid-sum table
  const uint32_t table_bytes = comp ? 64u * 32u * 4u : 0u;
  // Widest tile first (fewer, longer TMA boxes per byte moved), except for
  // calls with fewer (item, layer, channel) slabs than SMs: their tiles are
  // the only parallelism, so the narrowest tile that keeps rotation pairs
  // whole spreads them over the most SMs.
  const int n_ch_work = mode == MODE_RELOCATE_IN_PLACE ? 1 : n_ch_layout;
  const bool small_call = (int64_t)n_items * model->num_layers * n_ch_work < (int64_t)facts->sms;
  const int cands[4] = {256, 192, 128, 64};
  // Shape preference, measured on the three patched workloads: double-buffered
  // patch-factor slots with at most one trip through them per tile (K chunks
  // <= slots; the factor loads then keep pace with the canonical stream), then
  // as many canonical stages as fit (they carry the HBM stream), then the
  // widest factor chunks (whole rows of up to 128 bytes per TMA request).  A
  // second pass drops the first rule when nothing fits under it.
  const int u_max = use_patch ? (uv_env > 2 ? uv_env : 2) : 1;
  for (int pass = 0; pass < 2 && BN == 0; ++pass) {
    for (int ci = 0; ci < 4 && BN == 0; ++ci) {
      const int bn = cands[small_call ? 3 - ci : ci];
      if (bn_env && bn != bn_env) continue;
      if (D % bn != 0) continue;
      if (comp && bn % 128 != 0) continue;  // 128-column K boxes; 16-byte V code boxes
      bool whole = true;  // every rotate-half pair inside one column block
      for (int g = 0; g < n_groups; ++g)
        if (p.group_kind[g] > 0 && (g * 32) / bn != ((g + p.group_kind[g]) * 32) / bn) whole = false;
      if (!whole) continue;
      const uint32_t sb = (uint32_t)bn * (comp ? 384u : 256u);
      for (int s = 6; s >= 2 && BN == 0; --s) {
        if (st_env && s != st_env) continue;
        for (int ks = 1; ks <= (use_patch ? 4 : 1) && BN == 0; ks *= 2) {
          if (ks_env && use_patch && ks != ks_env) continue;
          if (use_patch && (rank / ks) % 16 != 0 && !(ks == 1 && rank == 8)) continue;  // whole K=16 steps
          for (int u = u_max; u >= 1 && BN == 0; --u) {
            if (uv_env && use_patch && u != uv_env) continue;
            if (pass == 0 && use_patch && !uv_env && !ks_env && (u < 2 || ks > u)) continue;
            const int kg = use_patch ? (rank / 8 / ks < 2 ? 2 : rank / 8 / ks) : 0;
            const uint32_t ub = use_patch ? (uint32_t)(BM + bn) * kg * 16u : 0u;
            const uint64_t need = (uint64_t)s * sb + (uint64_t)(use_patch ? u : 0) * ub + table_bytes +
                                  smem_extra_bytes(s, u, n_pairs);
            if (need > (uint64_t)facts->smem_optin) continue;
            BN = bn;
            stages = s;
            uv_slots = use_patch ? u : 0;
            ksplit = use_patch ? ks : 1;
            kg_alloc = kg;
            stage_bytes = sb;
            uv_slot_bytes = ub;
          }
        }
      }
    }
  }
  if (BN == 0) return fail(KAMERA_ERR_UNSUPPORTED, "no tile shape fits D = %d, rank %d", D, rank);
  const uint32_t smem = (uint32_t)stages * stage_bytes + (uint32_t)uv_slots * uv_slot_bytes + table_bytes +
                        smem_extra_bytes(stages, uv_slots, n_pairs);

  // ---- parameters ------------------------------------------------------------------------------------
  p.items = items;
  p.n_items = n_items;
  p.src_pool = (use_store || comp) ? 0 : 1;
  p.has_patches = use_patch ? 1 : 0;
  p.need_patch = mode == MODE_PATCH_IN_PLACE ? 1 : 0;
  p.rank = rank;
  p.ksplit = ksplit;
  p.ksteps = (rank / ksplit + 15) / 16;
  p.kg_alloc = kg_alloc;
  p.pool[0] = static_cast<uint16_t*>(pool->k);
  p.pool[1] = static_cast<uint16_t*>(pool->v);
  p.num_pages = pool->num_pages;
  p.page_size = pool->page_size;
  p.page_shift = __builtin_ctz((unsigned)pool->page_size);
  p.block_table = pool->block_table;
  p.n_seqs = pool->n_seqs;
  p.max_pages = pool->max_pages_per_seq;
  p.num_layers = model->num_layers;
  p.D = D;
  p.n_ch_layout = n_ch_layout;
  p.n_ch_work = n_ch_work;
  p.BN = BN;
  p.stages = stages;
  p.uv_slots = uv_slots;
  p.seg_rows = pool->page_size < BM ? pool->page_size : BM;
  p.seg_shift = __builtin_ctz((unsigned)p.seg_rows);
  p.rotate = mode == MODE_PATCH_IN_PLACE ? 0 : 1;
  p.frame = model->patch_frame;
  p.n_pairs = n_pairs;
  p.sec_end0 = sec_sum ? sec[0] : n_pairs;
  p.sec_end1 = sec_sum ? sec[0] + sec[1] : n_pairs;
  p.section_delta = sec_sum ? model->section_delta : nullptr;
  p.stage_bytes = stage_bytes;
  p.u_bytes = use_patch ? (uint32_t)BM * kg_alloc * 16u : 0u;
  p.v_bytes = use_patch ? (uint32_t)BN * kg_alloc * 16u : 0u;
  uint32_t tc = 32;
  while (tc < 2u * (uint32_t)BN) tc <<= 1;
  p.tmem_cols = tc;
  p.err_flag = err_flag;
  p.wait_limit_ns = tune.wait_limit_ns > 0 ? (uint64_t)tune.wait_limit_ns : WAIT_LIMIT_NS;
  p.test_unarm = tune.test_unarm_first_stage ? 1 : 0;
  if (mode == MODE_RELOCATE_IN_PLACE) {
    // only the column blocks that hold rotated groups change
    int lo = D / BN, hi = -1;
    for (int g = 0; g < n_groups; ++g)
      if (p.group_kind[g] != GK_PLAIN) {
        lo = (g * 32) / BN < lo ? (g * 32) / BN : lo;
        hi = (g * 32) / BN > hi ? (g * 32) / BN : hi;
      }
    p.cb_first = lo;
    p.n_cb = hi - lo + 1;
  } else {
    p.cb_first = 0;
    p.n_cb = D / BN;
  }

  // ---- tensor maps --------------------------------------------------------------------------------------
  if (use_store) {
    p.store_off = store->offset;
    p.store_len = store->len;
    p.store_elems = store->n_elems;
    p.n_chunks = store->n_chunks;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)(store_rows > 0 ? store_rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BOX_COLS, (cuuint32_t)BM};
    if (kamera_status st = encode(&p.src_map, store->data, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                                  "chunk store"))
      return st;
  }
  {
    for (int ch = 0; ch < p.n_ch_work; ++ch) {
      const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)pool_rows};
      const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
      const cuuint32_t box[2] = {(cuuint32_t)BOX_COLS, (cuuint32_t)p.seg_rows};
      if (kamera_status st = encode(&p.pool_map[ch], ch == 0 ? pool->k : pool->v, 2, dims, strides, box,
                                    CU_TENSOR_MAP_SWIZZLE_128B, "pool"))
        return st;
      const cuuint32_t box8[2] = {(cuuint32_t)BOX_COLS, 8u};
      if (kamera_status st = encode(&p.pool_map8[ch], ch == 0 ? pool->k : pool->v, 2, dims, strides, box8,
                                    CU_TENSOR_MAP_SWIZZLE_128B, "pool (8-row boxes)"))
        return st;
    }
  }
  if (comp) {
    const Codebook& cb = codebook();
    p.comp_row_offset = cstore->row_offset;
    p.comp_len = cstore->len;
    p.k_scale = cstore->k_scale;
    p.v_norm = cstore->v_norm;
    p.comp_rows = cstore->n_rows;
    p.n_chunks = cstore->n_chunks;
    p.head_dim = model->head_dim;
    p.out_bytes = (uint32_t)BN * 256u;
    p.table_bytes = table_bytes;
    for (int i = 0; i < 64; ++i) p.pair_sum[i] = cb.pair_sum[i];
    const cuuint64_t rows = (cuuint64_t)(cstore->n_rows > 0 ? cstore->n_rows : 1);
    const cuuint64_t kdims[2] = {(cuuint64_t)D, rows};
    const cuuint64_t kstrides[1] = {(cuuint64_t)D};
    const cuuint32_t kbox[2] = {128u, (cuuint32_t)BM};
    if (kamera_status st = encode(&p.kc_map, cstore->k_codes, 2, kdims, kstrides, kbox, CU_TENSOR_MAP_SWIZZLE_128B,
                                  "K codes", CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return st;
    const cuuint64_t vdims[2] = {(cuuint64_t)(3 * D / 8), rows};
    const cuuint64_t vstrides[1] = {(cuuint64_t)(3 * D / 8)};
    const cuuint32_t vbox[2] = {(cuuint32_t)(3 * BN / 8), (cuuint32_t)BM};
    if (kamera_status st = encode(&p.vc_map, cstore->v_codes, 2, vdims, vstrides, vbox, CU_TENSOR_MAP_SWIZZLE_NONE,
                                  "V codes", CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return st;
  }
  if (use_patch) {
    p.patch_off = patches->offset;
    p.patch_len = patches->len;
    p.patch_elems = patches->n_elems;
    p.n_patches = patches->n_patches;
    const int kw = rank / ksplit;  // K elements per chunk
    if (kw >= 16 && !comp) {  // (the compressed variant measured faster with core-matrix boxes)
      // whole chunk rows (2 kw = 32, 64 or 128 bytes) per TMA row, swizzled at that width: the
      // K-major layout tcgen05.mma reads with the matching swizzle mode
      p.uv_row_bytes = 2 * kw;
      const CUtensorMapSwizzle swz = kw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                     : (kw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
      const cuuint64_t dims[2] = {(cuuint64_t)rank, (cuuint64_t)(patch_rows > 0 ? patch_rows : 1)};
      const cuuint64_t strides[1] = {(cuuint64_t)rank * 2};
      const cuuint32_t ubox[2] = {(cuuint32_t)kw, (cuuint32_t)BM};
      const cuuint32_t vbox[2] = {(cuuint32_t)kw, (cuuint32_t)BN};
      if (kamera_status st = encode(&p.u_map, patches->data, 2, dims, strides, ubox, swz, "U")) return st;
      if (kamera_status st = encode(&p.v_map, patches->data, 2, dims, strides, vbox, swz, "V")) return st;
    } else {
      // rank 8 (16-byte rows) and the compressed variant: K-major core matrices (8 rows x 16 bytes)
      p.uv_row_bytes = 0;
      const cuuint64_t dims[3] = {8, (cuuint64_t)(patch_rows > 0 ? patch_rows : 1), (cuuint64_t)(rank / 8)};
      const cuuint64_t strides[2] = {(cuuint64_t)rank * 2, 16};
      const cuuint32_t ubox[3] = {8, (cuuint32_t)BM, (cuuint32_t)(rank / 8 / ksplit)};
      const cuuint32_t vbox[3] = {8, (cuuint32_t)BN, (cuuint32_t)(rank / 8 / ksplit)};
      if (kamera_status st = encode(&p.u_map, patches->data, 3, dims, strides, ubox, CU_TENSOR_MAP_SWIZZLE_NONE, "U"))
        return st;
      if (kamera_status st = encode(&p.v_map, patches->data, 3, dims, strides, vbox, CU_TENSOR_MAP_SWIZZLE_NONE, "V"))
        return st;
    }
  }

  // ---- launch ----------------------------------------------------------------------------------------------
  const void* fns[4] = {reinterpret_cast<const void*>(&reuse_kernel<false, false>),
                        reinterpret_cast<const void*>(&reuse_kernel<true, false>),
                        reinterpret_cast<const void*>(&reuse_kernel<false, true>),
                        reinterpret_cast<const void*>(&reuse_kernel<true, true>)};
  const int variant = (use_patch ? 1 : 0) + (comp ? 2 : 0);
  const void* fn = fns[variant];
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    bool& set = facts->attr_set[variant];
    if (!set) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, facts->smem_optin);
      if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      set = true;
    }
  }
  // Programmatic dependent launch: this grid may be scheduled while the
  // previous kernel on the stream drains; the kernel waits for it
  // (griddepcontrol.wait) before touching global memory.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tune.grid > 0 ? tune.grid : facts->sms));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = tune.no_pdl ? 0 : 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  switch (variant) {
    case 0: e = cudaLaunchKernelEx(&cfg, reuse_kernel<false, false>, p); break;
    case 1: e = cudaLaunchKernelEx(&cfg, reuse_kernel<true, false>, p); break;
    case 2: e = cudaLaunchKernelEx(&cfg, reuse_kernel<false, true>, p); break;
    default: e = cudaLaunchKernelEx(&cfg, reuse_kernel<true, true>, p); break;
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return KAMERA_OK;
}

// ---- compressed store encoder ---------------------------------------------------------------------

kamera_status compress_chunks(const kamera_model_desc* model, const kamera_chunk_store* src,
                              const kamera_compressed_store* dst, int32_t* err_flag, kamera_stream_t stream) {
  g_last_error.clear();
  if (!model || !src || !dst) return fail(KAMERA_ERR_NULL, "model, src or dst is NULL");
  if (model->family != KAMERA_MHA && model->family != KAMERA_GQA)
    return fail(model->family == KAMERA_MLA ? KAMERA_ERR_UNSUPPORTED : KAMERA_ERR_INVALID_ARG,
                "compressed store: family = %d (MHA/GQA served)", model->family);
  if (model->num_layers < 1 || model->num_kv_heads < 1)
    return fail(KAMERA_ERR_INVALID_ARG, "num_layers = %d, num_kv_heads = %d", model->num_layers,
                model->num_kv_heads);
  const int hd = model->head_dim;
  if (hd != 64 && hd != 128) return fail(KAMERA_ERR_UNSUPPORTED, "compressed store: head_dim = %d (64 or 128)", hd);
  const int D = model->num_kv_heads * hd;
  if (D % 128 != 0 || D > 32 * MAX_GROUPS)
    return fail(KAMERA_ERR_UNSUPPORTED, "compressed store: D = %d (a multiple of 128 up to %d)", D, 32 * MAX_GROUPS);
  if (src->n_chunks < 0 || dst->n_chunks != src->n_chunks)
    return fail(KAMERA_ERR_INVALID_ARG, "n_chunks: src %d, dst %d", src->n_chunks, dst->n_chunks);
  if (dst->n_rows < 0 || src->n_elems < 0 || dst->reserved != 0)
    return fail(KAMERA_ERR_INVALID_ARG, "sizes: src n_elems %lld, dst n_rows %lld", (long long)src->n_elems,
                (long long)dst->n_rows);
  if (src->n_chunks == 0) return KAMERA_OK;
  if (!src->data || !src->offset || !src->len || !dst->k_codes || !dst->k_scale || !dst->v_codes || !dst->v_norm ||
      !dst->row_offset || !dst->len)
    return fail(KAMERA_ERR_NULL, "a store pointer is NULL");
  if (!aligned16(src->data) || !aligned16(dst->k_codes) || !aligned16(dst->v_codes) ||
      (reinterpret_cast<uintptr_t>(dst->k_scale) & 3u) || (reinterpret_cast<uintptr_t>(dst->v_norm) & 3u))
    return fail(KAMERA_ERR_ALIGNMENT, "store data and codes must be 16-byte aligned");
  if (err_flag && (reinterpret_cast<uintptr_t>(err_flag) & 3u))
    return fail(KAMERA_ERR_ALIGNMENT, "err_flag must be 4-byte aligned");
  if (src->n_chunks > 65535) return fail(KAMERA_ERR_UNSUPPORTED, "n_chunks = %d (<= 65535)", src->n_chunks);
  int dev = 0;
  DeviceFacts* facts = nullptr;
  if (kamera_status st = device_facts(&dev, &facts)) return st;
  const Codebook& cb = codebook();
  compress::Args a;
  a.store = static_cast<const uint16_t*>(src->data);
  a.store_off = src->offset;
  a.store_len = src->len;
  a.store_elems = src->n_elems;
  a.k_codes = static_cast<int8_t*>(dst->k_codes);
  a.k_scale = dst->k_scale;
  a.v_codes = static_cast<uint8_t*>(dst->v_codes);
  a.v_norm = dst->v_norm;
  a.row_offset = dst->row_offset;
  a.len = dst->len;
  a.rows = dst->n_rows;
  a.n_chunks = src->n_chunks;
  a.L = model->num_layers;
  a.D = D;
  a.H = model->num_kv_heads;
  a.hd = hd;
  for (int k = 0; k < 7; ++k) a.thresholds[k] = cb.t[k];
  a.err_flag = err_flag;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  compress::k_scale_kernel<<<dim3((unsigned)a.L, (unsigned)a.n_chunks), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  // about four waves of 128-thread blocks, split across the chunks
  const int gx = (int)std::max<int64_t>(1, (int64_t)facts->sms * 16 / src->n_chunks);
  if (hd == 128)
    compress::encode_kernel<128><<<dim3((unsigned)gx, (unsigned)a.n_chunks), compress::THREADS, 0, s>>>(a);
  else
    compress::encode_kernel<64><<<dim3((unsigned)gx, (unsigned)a.n_chunks), compress::THREADS, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return KAMERA_OK;
}

// ---- patch formation -------------------------------------------------------------------------------

struct FactorShape {
  int kp, grid;
  int64_t work_per_cta;  // floats
};

kamera_status factor_validate(const kamera_factor_desc* d) {
  if (!d) return fail(KAMERA_ERR_NULL, "factor desc is NULL");
  if (d->n_slabs < 0) return fail(KAMERA_ERR_INVALID_ARG, "n_slabs = %d", d->n_slabs);
  if (d->T < 1 || d->T > 8192 || d->D < 1 || d->D > 2048)
    return fail(KAMERA_ERR_UNSUPPORTED, "slab %d x %d (T <= 8192, D <= 2048 served)", d->T, d->D);
  if (d->rank != 8 && d->rank != 16 && d->rank != 32 && d->rank != 64)
    return fail(KAMERA_ERR_INVALID_ARG, "rank = %d (8, 16, 32 or 64)", d->rank);
  const int k = d->rank + d->oversample;
  if (d->oversample < 0 || k > factor::KMAX)
    return fail(KAMERA_ERR_INVALID_ARG, "rank + oversample = %d (at most %d)", k, factor::KMAX);
  if (d->power_iters < 0 || d->power_iters > 8) return fail(KAMERA_ERR_INVALID_ARG, "power_iters = %d", d->power_iters);
  if (d->n_slabs > 1 && d->delta_stride < (int64_t)d->T * d->D)
    return fail(KAMERA_ERR_INVALID_ARG, "delta_stride < T*D");
  if (d->n_slabs > 0 && (!d->delta || !d->omega)) return fail(KAMERA_ERR_NULL, "delta or omega is NULL");
  return KAMERA_OK;
}

kamera_status factor_shape(const kamera_factor_desc* d, FactorShape* fs) {
  int dev = 0;
  DeviceFacts* facts = nullptr;
  if (kamera_status st = device_facts(&dev, &facts)) return st;
  const int k = d->rank + d->oversample;
  fs->kp = (k + 15) / 16 * 16;
  fs->grid = d->n_slabs < 2 * facts->sms ? d->n_slabs : 2 * facts->sms;  // two CTAs per SM
  fs->work_per_cta = (int64_t)fs->kp * (d->T + 2 * (int64_t)d->D);
  return KAMERA_OK;
}

// The tensor maps of the aligned instance's tall products (the table beside FactorMap).
kamera_status factor_maps(factor::FParams* f, int grid) {
  using namespace factor;
  const cuuint64_t T = (cuuint64_t)f->T, D = (cuuint64_t)f->D, k = (cuuint64_t)f->k, kp = (cuuint64_t)f->kp;
  const cuuint64_t m = (cuuint64_t)f->m, n = (cuuint64_t)f->n_slabs, g = (cuuint64_t)grid;
  const cuuint64_t slab = f->n_slabs > 1 ? (cuuint64_t)f->delta_stride : T * D;  // a single slab: any stride
  const cuuint64_t wpc = (cuuint64_t)f->work_per_cta;
  const float* Y = f->work;
  const float* Z = Y + kp * T;
  const float* Bw = Z + kp * D;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B, AT = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
  struct Spec {
    int idx;
    const void* base;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    CUtensorMapSwizzle swz;
    const char* what;
  };
  const Spec specs[] = {
      {MAP_DELTA_K, f->delta, {D, T, n}, {D * 4, slab * 4}, {32, 128, 1}, SW, "delta (K-major)"},
      {MAP_DELTA_MN, f->delta, {D, T, n}, {D * 4, slab * 4}, {32, 32, 1}, AT, "delta (M-major)"},
      {MAP_OMEGA_MN, f->omega, {k, D, 1}, {k * 4, k * D * 4}, {32, 32, 1}, AT, "omega"},
      {MAP_Y_K, Y, {T, kp, g}, {T * 4, wpc * 4}, {32, 64, 1}, SW, "Y (K-major)"},
      {MAP_Z_K, Z, {D, kp, g}, {D * 4, wpc * 4}, {32, 64, 1}, SW, "Z (K-major)"},
      {MAP_Y_MN, Y, {T, kp, g}, {T * 4, wpc * 4}, {32, 32, 1}, AT, "Y (M-major)"},
      {MAP_W_MN, Z, {m, kp, g}, {m * 4, wpc * 4}, {32, 32, 1}, AT, "W_m"},
      {MAP_B_MN, Bw, {D, kp, g}, {D * 4, wpc * 4}, {32, 32, 1}, AT, "B (M-major)"},
  };
  for (const Spec& sp : specs)
    if (kamera_status st = encode(&f->maps[sp.idx], sp.base, 3, sp.dims, sp.strides, sp.box, sp.swz, sp.what,
                                  CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return st;
  return KAMERA_OK;
}

// The aligned instance when the shapes and pointers allow it (the conditions of
// factor_kernel<true>), else the one with run-time fallbacks.
kamera_status launch_factor(const factor::FParams& fp, int grid, uint32_t smem, kamera_stream_t stream) {
  int dev = 0;
  DeviceFacts* facts = nullptr;
  if (kamera_status st = device_facts(&dev, &facts)) return st;
  {
    // the shared-memory limit is a function attribute of each device: raise it once per device
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!facts->factor_attr_set) {
      const int most = (int)factor::factor_smem_bytes(factor::KMAX, 64);
      cudaError_t e = factor::set_smem_limit_aligned(most);
      if (e == cudaSuccess) e = factor::set_smem_limit_general(most);
      if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      facts->factor_attr_set = true;
    }
  }
  const bool aligned = ((fp.T | fp.D | fp.k) & 3) == 0 && (fp.delta_stride & 3) == 0 &&
                       ((reinterpret_cast<uintptr_t>(fp.delta) | reinterpret_cast<uintptr_t>(fp.omega) |
                         reinterpret_cast<uintptr_t>(fp.work)) & 15u) == 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (aligned) {
    factor::FParams fa = fp;
    if (kamera_status st = factor_maps(&fa, grid)) return st;
    e = factor::launch_aligned(fa, grid, smem, s);
  } else {
    e = factor::launch_general(fp, grid, smem, s);
  }
  if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return KAMERA_OK;
}

kamera_status factor_workspace_size(const kamera_factor_desc* d, size_t* bytes) {
  g_last_error.clear();
  if (!bytes) return fail(KAMERA_ERR_NULL, "bytes is NULL");
  if (kamera_status st = factor_validate(d)) return st;
  FactorShape fs;
  if (kamera_status st = factor_shape(d, &fs)) return st;
  *bytes = (size_t)fs.grid * (size_t)fs.work_per_cta * sizeof(float);
  return KAMERA_OK;
}

kamera_status factor_patches(const kamera_factor_desc* d, void* u_out, void* v_out, int64_t out_stride,
                             void* workspace, size_t workspace_bytes, kamera_stream_t stream) {
  g_last_error.clear();
  if (kamera_status st = factor_validate(d)) return st;
  if (d->n_slabs == 0) return KAMERA_OK;
  if (!u_out || !v_out || !workspace) return fail(KAMERA_ERR_NULL, "u_out, v_out or workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || (reinterpret_cast<uintptr_t>(d->delta) & 15u) ||
      (reinterpret_cast<uintptr_t>(u_out) & 1u) || (reinterpret_cast<uintptr_t>(v_out) & 1u))
    return fail(KAMERA_ERR_ALIGNMENT, "workspace must be 256-byte aligned, delta 16-byte, outputs 2-byte");
  if (out_stride < (int64_t)d->rank * (d->T > d->D ? d->T : d->D) && d->n_slabs > 1)
    return fail(KAMERA_ERR_INVALID_ARG, "out_stride %lld overlaps consecutive slabs", (long long)out_stride);
  FactorShape fs;
  if (kamera_status st = factor_shape(d, &fs)) return st;
  if (workspace_bytes < (size_t)fs.grid * (size_t)fs.work_per_cta * sizeof(float))
    return fail(KAMERA_ERR_INVALID_ARG, "workspace of %zu bytes is too small", workspace_bytes);
  factor::FParams fp;
  fp.delta = d->delta;
  fp.delta_stride = d->delta_stride;
  fp.n_slabs = d->n_slabs;
  fp.T = d->T;
  fp.D = d->D;
  fp.m = d->rank;
  fp.k = d->rank + d->oversample;
  fp.kp = fs.kp;
  fp.power_iters = d->power_iters;
  fp.omega = d->omega;
  fp.u_out = static_cast<uint16_t*>(u_out);
  fp.v_out = static_cast<uint16_t*>(v_out);
  fp.out_stride = out_stride;
  fp.work = static_cast<float*>(workspace);
  fp.work_per_cta = fs.work_per_cta;
  const uint32_t smem = factor::factor_smem_bytes(fs.kp, d->rank);
  return launch_factor(fp, fs.grid, smem, stream);
}

kamera_status orbit_mean(const float* deltas, int32_t n, int64_t stride, int64_t n_elems, float* out,
                         kamera_stream_t stream) {
  g_last_error.clear();
  if (n < 1) return fail(KAMERA_ERR_INVALID_ARG, "n_orderings = %d", n);
  if (n_elems < 0) return fail(KAMERA_ERR_INVALID_ARG, "n_elems = %lld", (long long)n_elems);
  if (n > 1 && stride < n_elems) return fail(KAMERA_ERR_INVALID_ARG, "ordering_stride < n_elems");
  if (n_elems == 0) return KAMERA_OK;
  if (!deltas || !out) return fail(KAMERA_ERR_NULL, "deltas or out is NULL");
  if ((reinterpret_cast<uintptr_t>(deltas) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u))
    return fail(KAMERA_ERR_ALIGNMENT, "deltas and out must be 4-byte aligned");
  const char* lo_in = reinterpret_cast<const char*>(deltas);
  const char* hi_in = lo_in + ((int64_t)(n - 1) * stride + n_elems) * 4;
  const char* lo_out = reinterpret_cast<const char*>(out);
  if (lo_out < hi_in && lo_in < lo_out + n_elems * 4) return fail(KAMERA_ERR_INVALID_ARG, "out overlaps the inputs");
  int dev = 0;
  DeviceFacts* facts = nullptr;
  if (kamera_status st = device_facts(&dev, &facts)) return st;
  const int64_t want = (n_elems / 4 + 255) / 256;
  const int grid = (int)(want < 8LL * facts->sms ? (want > 0 ? want : 1) : 8LL * facts->sms);
  factor::orbit_mean_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(deltas, n, stride, n_elems, out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return KAMERA_OK;
}

// ---- patch formation without a caller workspace --------------------------------------------------
// Callers that cannot allocate get their scratch from this fixed array.  In
// host code its name is only a host-side stand-in: the device address comes
// from cudaGetSymbolAddress, looked up once per device with that device
// current.
constexpr size_t kStaticScratchFloats = KAMERA_FACTOR_STATIC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_factor_scratch[kStaticScratchFloats];
float* g_scratch_addr[kMaxDevices] = {};

kamera_status static_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(KAMERA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(KAMERA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_factor_scratch);
    if (e != cudaSuccess || !ptr)
      return fail(KAMERA_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = static_cast<float*>(ptr);
  }
  *out = g_scratch_addr[dev];
  return KAMERA_OK;
}

kamera_status factor_patches_noalloc(const kamera_factor_desc* d, void* u_out, void* v_out, int64_t out_stride,
                                     kamera_stream_t stream) {
  g_last_error.clear();
  if (kamera_status st = factor_validate(d)) return st;
  if (d->n_slabs == 0) return KAMERA_OK;
  if (!u_out || !v_out) return fail(KAMERA_ERR_NULL, "u_out or v_out is NULL");
  if ((reinterpret_cast<uintptr_t>(d->delta) & 15u) || (reinterpret_cast<uintptr_t>(u_out) & 1u) ||
      (reinterpret_cast<uintptr_t>(v_out) & 1u))
    return fail(KAMERA_ERR_ALIGNMENT, "delta must be 16-byte aligned, outputs 2-byte");
  if (out_stride < (int64_t)d->rank * (d->T > d->D ? d->T : d->D) && d->n_slabs > 1)
    return fail(KAMERA_ERR_INVALID_ARG, "out_stride %lld overlaps consecutive slabs", (long long)out_stride);
  FactorShape fs;
  if (kamera_status st = factor_shape(d, &fs)) return st;
  if ((size_t)fs.work_per_cta > kStaticScratchFloats)
    return fail(KAMERA_ERR_UNSUPPORTED,
                "one %d x %d slab at k = %d needs %lld bytes of scratch; the static region holds %zu bytes",
                d->T, d->D, fs.kp, (long long)fs.work_per_cta * 4, (size_t)KAMERA_FACTOR_STATIC_SCRATCH_BYTES);
  const int64_t fit = (int64_t)(kStaticScratchFloats / (size_t)fs.work_per_cta);
  const int grid = (int)(fit < fs.grid ? fit : fs.grid);
  float* scratch = nullptr;
  if (kamera_status st = static_scratch(&scratch)) return st;
  factor::FParams fp;
  fp.delta = d->delta;
  fp.delta_stride = d->delta_stride;
  fp.n_slabs = d->n_slabs;
  fp.T = d->T;
  fp.D = d->D;
  fp.m = d->rank;
  fp.k = d->rank + d->oversample;
  fp.kp = fs.kp;
  fp.power_iters = d->power_iters;
  fp.omega = d->omega;
  fp.u_out = static_cast<uint16_t*>(u_out);
  fp.v_out = static_cast<uint16_t*>(v_out);
  fp.out_stride = out_stride;
  fp.work = scratch;
  fp.work_per_cta = fs.work_per_cta;
  const uint32_t smem = factor::factor_smem_bytes(fs.kp, d->rank);
  return launch_factor(fp, grid, smem, stream);
}

}  // namespace
}  // namespace kamera

extern "C" {

kamera_status kamera_factor_patches_noalloc(const kamera_factor_desc* desc, void* u_out, void* v_out,
                                            int64_t out_stride, kamera_stream_t stream) {
  return kamera::factor_patches_noalloc(desc, u_out, v_out, out_stride, stream);
}

kamera_status kamera_orbit_mean(const float* deltas, int32_t n_orderings, int64_t ordering_stride, int64_t n_elems,
                                float* out, kamera_stream_t stream) {
  return kamera::orbit_mean(deltas, n_orderings, ordering_stride, n_elems, out, stream);
}

kamera_status kamera_factor_workspace_size(const kamera_factor_desc* desc, size_t* bytes) {
  return kamera::factor_workspace_size(desc, bytes);
}

kamera_status kamera_factor_patches(const kamera_factor_desc* desc, void* u_out, void* v_out, int64_t out_stride,
                                    void* workspace, size_t workspace_bytes, kamera_stream_t stream) {
  return kamera::factor_patches(desc, u_out, v_out, out_stride, workspace, workspace_bytes, stream);
}

kamera_status kamera_reuse_batched(const kamera_model_desc* model, const kamera_chunk_store* store,
                                   const kamera_patch_store* patches, const kamera_reuse_item* items,
                                   int32_t n_items, const kamera_paged_pool* pool, int32_t* err_flag,
                                   kamera_stream_t stream) {
  return kamera::launch(kamera::MODE_REUSE, model, store, patches, items, n_items, pool, err_flag, stream);
}

kamera_status kamera_relocate(const kamera_model_desc* model, const kamera_chunk_store* store,
                              const kamera_reuse_item* items, int32_t n_items, const kamera_paged_pool* pool,
                              int32_t* err_flag, kamera_stream_t stream) {
  return kamera::launch(store ? kamera::MODE_REUSE : kamera::MODE_RELOCATE_IN_PLACE, model, store, nullptr, items,
                        n_items, pool, err_flag, stream);
}

kamera_status kamera_apply_patch(const kamera_model_desc* model, const kamera_patch_store* patches,
                                 const kamera_reuse_item* items, int32_t n_items, const kamera_paged_pool* pool,
                                 int32_t* err_flag, kamera_stream_t stream) {
  return kamera::launch(kamera::MODE_PATCH_IN_PLACE, model, nullptr, patches, items, n_items, pool, err_flag,
                        stream);
}

kamera_status kamera_v_codebook(float centroids[8], float thresholds[7]) {
  const kamera::Codebook& cb = kamera::codebook();
  if (centroids) memcpy(centroids, cb.c, sizeof cb.c);
  if (thresholds) memcpy(thresholds, cb.t, sizeof cb.t);
  return KAMERA_OK;
}

kamera_status kamera_compress_chunks(const kamera_model_desc* model, const kamera_chunk_store* src,
                                     const kamera_compressed_store* dst, int32_t* err_flag, kamera_stream_t stream) {
  return kamera::compress_chunks(model, src, dst, err_flag, stream);
}

kamera_status kamera_reuse_compressed(const kamera_model_desc* model, const kamera_compressed_store* store,
                                      const kamera_patch_store* patches, const kamera_reuse_item* items,
                                      int32_t n_items, const kamera_paged_pool* pool, int32_t* err_flag,
                                      kamera_stream_t stream) {
  if (!store) {
    kamera::g_last_error = "compressed store is NULL";
    return KAMERA_ERR_NULL;
  }
  return kamera::launch(kamera::MODE_REUSE, model, nullptr, patches, items, n_items, pool, err_flag, stream, store);
}

const char* kamera_status_string(kamera_status status) {
  switch (status) {
    case KAMERA_OK: return "KAMERA_OK";
    case KAMERA_ERR_NULL: return "KAMERA_ERR_NULL";
    case KAMERA_ERR_INVALID_ARG: return "KAMERA_ERR_INVALID_ARG";
    case KAMERA_ERR_UNSUPPORTED: return "KAMERA_ERR_UNSUPPORTED";
    case KAMERA_ERR_ALIGNMENT: return "KAMERA_ERR_ALIGNMENT";
    case KAMERA_ERR_CUDA: return "KAMERA_ERR_CUDA";
  }
  return "KAMERA_ERR_UNKNOWN";
}

const char* kamera_last_error(void) { return kamera::g_last_error.c_str(); }

kamera_status kamera_set_launch_tuning(const kamera_launch_tuning* tuning) { return kamera::set_tuning(tuning); }

kamera_status kamera_get_launch_tuning(kamera_launch_tuning* tuning) {
  if (!tuning) {
    kamera::g_last_error = "tuning is NULL";
    return KAMERA_ERR_NULL;
  }
  *tuning = kamera::current_tuning();
  return KAMERA_OK;
}

int32_t kamera_abi_version(void) { return KAMERA_ABI_VERSION; }

}  // extern "C"
