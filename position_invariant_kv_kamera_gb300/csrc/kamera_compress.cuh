// kamera_compress.cuh -- encoder of the compressed canonical store (sm_103a).
//
// PolyKV (gist.science summary), §2B, asymmetric compression: K as int8 with
// one linear scale per tensor; V at 3 bits per coordinate by TurboQuant MSE
// (rotate by a fast Walsh-Hadamard transform so the coordinates approach
// N(0,1), map each to the nearest Lloyd-Max centroid of N(0,1)).
//
// Format (include/kamera.h, kamera_compressed_store): chunk c, layer l, token
// t is store row row_offset[c] + l*T + t.  K: int8 codes [rows][D] and one
// scale s = max|x| / 127 per (chunk, layer), code rint(x / s) in [-127, 127].
// V: per head row of d = head_dim values, ||x|| (fp32) and 3d bits of codes;
// 6-bit field i (i < d/2) = code[i] | code[i + d/2] << 3 at bit 6i.  The code
// of coordinate e is the number of codebook thresholds <= (H x)_e / ||x||.
//
// Every decision is taken in fp32 in one fixed order of operations (part of
// the format, so that any conforming encoder gives the same bytes): the
// transform's butterflies level by level with strides 1, 2, 4, ...; the sum
// of squares in index order with fused multiply-add; IEEE division and square
// root.  The explicit __f*_rn intrinsics keep the compiler from contracting or
// reordering any of them.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "kamera.h"

namespace kamera {
namespace compress {

constexpr int THREADS = 128;

struct Args {
  const uint16_t* store;     // bf16 chunk store
  const int64_t* store_off;  // [n_chunks] element offsets
  const int32_t* store_len;  // [n_chunks]
  int64_t store_elems;
  int8_t* k_codes;           // [rows][D]
  float* k_scale;            // [n_chunks][L]
  uint8_t* v_codes;          // [rows][H][3*hd/8]
  float* v_norm;             // [rows][H]
  const int64_t* row_offset; // [n_chunks]
  const int32_t* len;        // [n_chunks]
  int64_t rows;
  int32_t n_chunks, L, D, H, hd;
  float thresholds[7];
  int32_t* err_flag;
};

// Error bits of chunk c (0 = it can be encoded).
__device__ __forceinline__ int32_t chunk_check(const Args& a, int32_t c) {
  const int64_t T = a.store_len[c];
  if (T < 0 || a.len[c] != T) return KAMERA_EFLAG_LEN;
  const int64_t off = a.store_off[c];
  if (off < 0 || off % a.D != 0 || off + (int64_t)a.L * 2 * T * a.D > a.store_elems) return KAMERA_EFLAG_CHUNK_OOB;
  const int64_t r0 = a.row_offset[c];
  if (r0 < 0 || r0 + (int64_t)a.L * T > a.rows) return KAMERA_EFLAG_CHUNK_OOB;
  return 0;
}

// K scale of (chunk blockIdx.y, layer blockIdx.x): max|x| / 127.
__global__ void __launch_bounds__(256) k_scale_kernel(const Args a) {
  const int32_t c = blockIdx.y, l = blockIdx.x;
  const int32_t bad = chunk_check(a, c);
  if (bad) {
    if (threadIdx.x == 0 && l == 0 && a.err_flag) atomicOr(a.err_flag, bad);
    return;
  }
  const int64_t T = a.store_len[c];
  const int64_t n = T * a.D;  // a multiple of 8
  const uint4* k = reinterpret_cast<const uint4*>(a.store + a.store_off[c] + (int64_t)l * 2 * n);
  float amax = 0.0f;
  for (int64_t i = threadIdx.x; i < n / 8; i += blockDim.x) {
    const uint4 v = __ldcs(k + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, part[w]);
    a.k_scale[(int64_t)c * a.L + l] = __fdiv_rn(amax, 127.0f);
  }
}

// One (chunk blockIdx.y, layer, token, head) per thread: that head's K codes
// and its V codes and norm.
template <int HD>
__global__ void __launch_bounds__(THREADS) encode_kernel(const Args a) {
  constexpr int NW = 3 * HD / 32;  // code words per head row
  const int32_t c = blockIdx.y;
  if (chunk_check(a, c)) return;
  const int64_t T = a.store_len[c];
  const int64_t units = (int64_t)a.L * T * a.H;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int32_t h = (int32_t)(u % a.H);
    const int64_t lt = u / a.H;  // l * T + t
    const int32_t l = (int32_t)(lt / T);
    const int64_t t = lt - (int64_t)l * T;
    const int64_t row = a.row_offset[c] + lt;
    const uint16_t* kx = a.store + a.store_off[c] + (((int64_t)l * 2 + 0) * T + t) * a.D + (int64_t)h * HD;
    const uint16_t* vx = a.store + a.store_off[c] + (((int64_t)l * 2 + 1) * T + t) * a.D + (int64_t)h * HD;

    // ---- K: q = rint(x / s), clamped to [-127, 127] ----
    const float s = a.k_scale[(int64_t)c * a.L + l];
    int8_t* kq = a.k_codes + row * a.D + (int64_t)h * HD;
    for (int e0 = 0; e0 < HD; e0 += 16) {
      const uint4 v0 = __ldcs(reinterpret_cast<const uint4*>(kx + e0));
      const uint4 v1 = __ldcs(reinterpret_cast<const uint4*>(kx + e0 + 8));
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t q[4] = {0, 0, 0, 0};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t bits = (e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
        int32_t qi = 0;
        if (s != 0.0f) {
          qi = __float2int_rn(__fdiv_rn(__uint_as_float(bits), s));
          qi = qi > 127 ? 127 : (qi < -127 ? -127 : qi);
        }
        q[e >> 2] |= ((uint32_t)qi & 0xFFu) << (8 * (e & 3));
      }
      *reinterpret_cast<uint4*>(kq + e0) = make_uint4(q[0], q[1], q[2], q[3]);
    }

    // ---- V: ||x||, w = H x, code = #{k : t_k <= w_e / ||x||} ----
    float x[HD];
#pragma unroll
    for (int e0 = 0; e0 < HD; e0 += 8) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(vx + e0));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[e0 + 2 * j] = __uint_as_float(w[j] << 16);
        x[e0 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < HD; ++e) acc = __fmaf_rn(x[e], x[e], acc);
    const float nr = __fsqrt_rn(acc);
#pragma unroll
    for (int hs = 1; hs < HD; hs <<= 1)
#pragma unroll
      for (int i = 0; i < HD; i += 2 * hs)
#pragma unroll
        for (int j = i; j < i + hs; ++j) {
          const float p = x[j], q = x[j + hs];
          x[j] = __fadd_rn(p, q);
          x[j + hs] = __fsub_rn(p, q);
        }
    uint32_t words[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) words[k] = 0;
#pragma unroll
    for (int e = 0; e < HD; ++e) {
      uint32_t code = 0;
      if (nr > 0.0f) {
        const float z = __fdiv_rn(x[e], nr);
#pragma unroll
        for (int k = 0; k < 7; ++k) code += (a.thresholds[k] <= z) ? 1u : 0u;
      }
      // the 3-bit group of coordinate e starts at a multiple of 3 and may straddle two words
      const int bit = 6 * (e % (HD / 2)) + (e < HD / 2 ? 0 : 3);
      words[bit >> 5] |= code << (bit & 31);
      if ((bit & 31) > 29) words[(bit >> 5) + 1] |= code >> (32 - (bit & 31));
    }
    uint8_t* vc = a.v_codes + (row * a.H + h) * (3 * HD / 8);
    if (HD == 128) {
#pragma unroll
      for (int k = 0; k < NW / 4; ++k)
        *reinterpret_cast<uint4*>(vc + 16 * k) =
            make_uint4(words[4 * k], words[4 * k + 1], words[4 * k + 2], words[4 * k + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < NW / 2; ++k) *reinterpret_cast<uint2*>(vc + 8 * k) = make_uint2(words[2 * k], words[2 * k + 1]);
    }
    a.v_norm[row * a.H + h] = nr;
  }
}

}  // namespace compress
}  // namespace kamera
