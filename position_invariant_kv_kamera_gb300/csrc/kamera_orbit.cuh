// kamera_orbit.cuh -- the orbit deficit on the GPU.
//
// Kamera: Unified Position-Invariant Multimodal KV Cache for Training-Free
// Reuse, §3 (orbit patch): the patch of a chunk that appears at varying places
// is formed from the deficit averaged over the orderings it was measured under.
// This kernel takes n sampled deficits (one fp32 array per ordering, the same
// shape) and writes their element-wise mean; its rank-m factors then come from
// patch formation like any other deficit.
#pragma once
#include <stdint.h>

namespace kamera {
namespace factor {

// Mean of n sampled deficits, element-wise, fp32, terms added in index order.
// Streaming: 16-byte loads when every row start is 16-byte aligned.
__global__ void orbit_mean_kernel(const float* __restrict__ d, int n, int64_t stride, int64_t n_elems,
                                  float* __restrict__ out) {
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(d) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0 &&
                   (stride & 3) == 0;
  const float fn = (float)n;
  if (vec) {
    const int64_t n4 = n_elems / 4;
    for (int64_t e = t0; e < n4; e += nthreads) {
      float4 s = __ldcs(reinterpret_cast<const float4*>(d) + e);
      for (int j = 1; j < n; ++j) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(d + (int64_t)j * stride) + e);
        s.x += x.x;
        s.y += x.y;
        s.z += x.z;
        s.w += x.w;
      }
      __stcs(reinterpret_cast<float4*>(out) + e, make_float4(__fdiv_rn(s.x, fn), __fdiv_rn(s.y, fn),
                                                            __fdiv_rn(s.z, fn), __fdiv_rn(s.w, fn)));
    }
    for (int64_t e = n4 * 4 + t0; e < n_elems; e += nthreads) {
      float s = d[e];
      for (int j = 1; j < n; ++j) s += d[(int64_t)j * stride + e];
      out[e] = __fdiv_rn(s, fn);
    }
  } else {
    for (int64_t e = t0; e < n_elems; e += nthreads) {
      float s = d[e];
      for (int j = 1; j < n; ++j) s += d[(int64_t)j * stride + e];
      out[e] = __fdiv_rn(s, fn);
    }
  }
}

}  // namespace factor
}  // namespace kamera
