// kamera_factor.cuh -- patch formation on the GPU: rank-m factors of a
// conditioning deficit.
//
// Kamera: Unified Position-Invariant Multimodal KV Cache for Training-Free
// Reuse, §2 "Patch application": the patch is computed once, from the deficit
// Delta = KV(B|A) - KV(B|empty) of one conditioned forward pass, by an SVD that
// keeps the top-m factors.  Given Delta (one [T][D] fp32 slab per patch, layer
// and channel) this kernel writes U_m [T][m] and V_m [D][m] (bf16) with
// U_m V_m^T the rank-m truncation of Delta, in the patch-store layout that the
// reuse kernel reads.
//
// Method: the randomized range finder with subspace iteration of Halko,
// Martinsson & Tropp ("Finding structure with randomness", SIAM Review 2011,
// Algorithms 4.4 and 5.1), all in fp32:
//   Y = Delta Omega (Omega [D][k] Gaussian, k = m + oversampling, an input);
//   Q = orth(Y);  q times: Z = orth(Delta^T Q), Q = orth(Delta Z);
//   B = Q^T Delta  [k][D];  C = B B^T = W Lambda W^T (cyclic Jacobi);
//   U_m = Q W_m (orthonormal columns),  V_m = B^T W_m (carries Sigma).
// orth() is classical Gram-Schmidt applied twice per column; a column whose
// remainder falls below 1e-4 of its norm is dropped (set to zero), so deficits
// of rank below k are handled exactly.
//
// One CTA (256 threads) per slab at a time; each CTA owns a workspace region
// (Y [k][T], Z [k][D], B [k][D], column-major panels) in global memory.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace kamera {
namespace factor {

constexpr int THREADS = 256;
constexpr int KMAX = 96;   // k = m + oversampling, padded to a multiple of 16
constexpr int GT = 64;     // GEMM tile (rows and columns)
constexpr int GK = 16;     // GEMM K step
constexpr int MAX_SWEEPS = 20;

struct FParams {
  const float* delta;    // [n_slabs][T][D]
  int64_t delta_stride;  // elements between slabs
  int32_t n_slabs, T, D, m, k, kp, power_iters;
  const float* omega;    // [D][k]
  uint16_t* u_out;       // slab s: u_out + s*out_stride, [T][m] bf16
  uint16_t* v_out;       // slab s: v_out + s*out_stride, [D][m] bf16
  int64_t out_stride;
  float* work;           // per CTA: work + blockIdx.x * work_per_cta
  int64_t work_per_cta;  // floats
};

// ---- CTA-wide fp32 GEMM: C(i,j) = sum_l A(i,l) B(l,j), arbitrary strides --------------
// Element (i,l) of A is A[i*a_rs + l*a_cs], and so on.  Tiles of 64x64, K step
// 16, 256 threads each owning a 4x4 block.  Out-of-range elements read as 0.
template <typename OutT>
__device__ void gemm(int M, int N, int K, const float* A, int64_t a_rs, int64_t a_cs, const float* B, int64_t b_rs,
                     int64_t b_cs, OutT* C, int64_t c_rs, int64_t c_cs, float* sA, float* sB) {
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  for (int i0 = 0; i0 < M; i0 += GT) {
    for (int j0 = 0; j0 < N; j0 += GT) {
      float acc[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
      for (int l0 = 0; l0 < K; l0 += GK) {
        // sA[l][i] (16 x 64), sB[l][j] (16 x 64); read along the contiguous dimension
        for (int e = tid; e < GK * GT; e += THREADS) {
          int i, l;
          if (a_cs == 1) { l = e % GK; i = e / GK; } else { i = e % GT; l = e / GT; }
          const int gi = i0 + i, gl = l0 + l;
          sA[l * GT + i] = (gi < M && gl < K) ? A[gi * a_rs + gl * a_cs] : 0.f;
          int j, l2;
          if (b_rs == 1) { l2 = e % GK; j = e / GK; } else { j = e % GT; l2 = e / GT; }
          const int gj = j0 + j, gl2 = l0 + l2;
          sB[l2 * GT + j] = (gj < N && gl2 < K) ? B[gl2 * b_rs + gj * b_cs] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int l = 0; l < GK; ++l) {
          float a[4], b[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            a[q] = sA[l * GT + ty * 4 + q];
            b[q] = sB[l * GT + tx * 4 + q];
          }
#pragma unroll
          for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
        }
        __syncthreads();
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int gi = i0 + ty * 4 + x, gj = j0 + tx * 4 + y;
          if (gi < M && gj < N) {
            if constexpr (sizeof(OutT) == 2) {
              __nv_bfloat16 h = __float2bfloat16_rn(acc[x][y]);
              C[gi * c_rs + gj * c_cs] = *reinterpret_cast<uint16_t*>(&h);
            } else {
              C[gi * c_rs + gj * c_cs] = acc[x][y];
            }
          }
        }
    }
  }
  __syncthreads();
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < THREADS / 32; ++i) s += red[i];
  return s;
}

// Orthonormalise the k columns (length n, column j at X + j*n) in place by
// classical Gram-Schmidt applied twice; dependent columns become zero.
__device__ void orth_cgs2(float* X, int n, int k, float* coef, float* red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int j = 0; j < k; ++j) {
    float* v = X + (int64_t)j * n;
    float n0 = 0.f;
    for (int t = tid; t < n; t += THREADS) n0 += v[t] * v[t];
    n0 = sqrtf(block_sum(n0, red));
    for (int pass = 0; pass < 2 && j > 0; ++pass) {
      // coef[l] = <q_l, v>, one warp per column l
      for (int l = warp; l < j; l += THREADS / 32) {
        const float* ql = X + (int64_t)l * n;
        float s = 0.f;
        for (int t = lane; t < n; t += 32) s += ql[t] * v[t];
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
        if (lane == 0) coef[l] = s;
      }
      __syncthreads();
      for (int t = tid; t < n; t += THREADS) {
        float s = v[t];
        for (int l = 0; l < j; ++l) s -= coef[l] * X[(int64_t)l * n + t];
        v[t] = s;
      }
      __syncthreads();
    }
    float nr = 0.f;
    for (int t = tid; t < n; t += THREADS) nr += v[t] * v[t];
    nr = sqrtf(block_sum(nr, red));
    const float scale = (nr > 1e-4f * n0 && nr > 0.f) ? 1.f / nr : 0.f;
    for (int t = tid; t < n; t += THREADS) v[t] *= scale;
    __syncthreads();
  }
}

// Cyclic Jacobi eigen-decomposition of the symmetric kp x kp matrix C (row
// major, in shared memory) with the parallel (round-robin tournament) order:
// each round rotates kp/2 disjoint planes at once.  On return the diagonal of
// C holds the eigenvalues and the columns of W the eigenvectors.
__device__ void jacobi_eig(float* C, float* W, int kp, float* rot, float* red) {
  const int tid = threadIdx.x;
  for (int e = tid; e < kp * kp; e += THREADS) W[e] = (e / kp == e % kp) ? 1.f : 0.f;
  __syncthreads();
  const int half = kp / 2;
  for (int sweep = 0; sweep < MAX_SWEEPS; ++sweep) {
    float off = 0.f, tot = 0.f;
    for (int e = tid; e < kp * kp; e += THREADS) {
      const float x = C[e];
      tot += x * x;
      if (e / kp != e % kp) off += x * x;
    }
    off = block_sum(off, red);
    tot = block_sum(tot, red);
    if (off <= 1e-12f * tot || tot == 0.f) break;
    for (int round = 0; round < kp - 1; ++round) {
      // pair i: players (i, kp-1-i) of the rotated ring; player 0 stays fixed
      if (tid < half) {
        int a = tid == 0 ? 0 : 1 + (tid - 1 + round) % (kp - 1);
        int b = 1 + (kp - 2 - tid + round) % (kp - 1);
        int p = min(a, b), q = max(a, b);
        const float app = C[p * kp + p], aqq = C[q * kp + q], apq = C[p * kp + q];
        float c = 1.f, s = 0.f;
        if (apq != 0.f && fabsf(apq) > 1e-30f) {
          const float zeta = (aqq - app) / (2.f * apq);
          const float t = copysignf(1.f, zeta) / (fabsf(zeta) + sqrtf(1.f + zeta * zeta));
          c = rsqrtf(1.f + t * t);
          s = c * t;
        }
        rot[4 * tid + 0] = (float)p;
        rot[4 * tid + 1] = (float)q;
        rot[4 * tid + 2] = c;
        rot[4 * tid + 3] = s;
      }
      __syncthreads();
      // rows p, q of C  (C <- J^T C)
      for (int e = tid; e < half * kp; e += THREADS) {
        const int i = e / kp, j = e % kp;
        const int p = (int)rot[4 * i], q = (int)rot[4 * i + 1];
        const float c = rot[4 * i + 2], s = rot[4 * i + 3];
        const float xp = C[p * kp + j], xq = C[q * kp + j];
        C[p * kp + j] = c * xp - s * xq;
        C[q * kp + j] = s * xp + c * xq;
      }
      __syncthreads();
      // columns p, q of C and of W  (C <- C J, W <- W J)
      for (int e = tid; e < half * kp; e += THREADS) {
        const int i = e / kp, j = e % kp;
        const int p = (int)rot[4 * i], q = (int)rot[4 * i + 1];
        const float c = rot[4 * i + 2], s = rot[4 * i + 3];
        float xp = C[j * kp + p], xq = C[j * kp + q];
        C[j * kp + p] = c * xp - s * xq;
        C[j * kp + q] = s * xp + c * xq;
        xp = W[j * kp + p];
        xq = W[j * kp + q];
        W[j * kp + p] = c * xp - s * xq;
        W[j * kp + q] = s * xp + c * xq;
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1) factor_kernel(const __grid_constant__ FParams p) {
  extern __shared__ __align__(16) float fsm[];
  float* sA = fsm;                       // GT*GK
  float* sB = sA + GT * GK;              // GT*GK
  float* C = sB + GT * GK;               // kp*kp
  float* W = C + KMAX * KMAX;            // kp*kp
  float* Ws = W + KMAX * KMAX;           // kp*m: sorted leading eigenvectors
  float* coef = Ws + KMAX * 64;          // KMAX
  float* rot = coef + KMAX;              // 4 * KMAX/2
  float* red = rot + 2 * KMAX;           // 32
  int* perm = reinterpret_cast<int*>(red + 32);  // KMAX

  const int T = p.T, D = p.D, k = p.k, kp = p.kp, m = p.m;
  float* Y = p.work + blockIdx.x * p.work_per_cta;  // [kp][T] column-major
  float* Z = Y + (int64_t)kp * T;                   // [kp][D]
  float* B = Z + (int64_t)kp * D;                   // [kp][D]: row i of B contiguous

  // rows k..kp-1 of B are never written: keep them zero for the V_m product
  for (int64_t e = (int64_t)k * D + threadIdx.x; e < (int64_t)kp * D; e += THREADS) B[e] = 0.f;
  for (int s = blockIdx.x; s < p.n_slabs; s += gridDim.x) {
    const float* A = p.delta + (int64_t)s * p.delta_stride;  // [T][D]
    // Y = Delta Omega (columns k..kp-1 stay zero)
    for (int64_t e = threadIdx.x; e < (int64_t)kp * T; e += THREADS) Y[e] = 0.f;
    __syncthreads();
    gemm<float>(T, k, D, A, D, 1, p.omega, k, 1, Y, 1, T, sA, sB);
    orth_cgs2(Y, T, k, coef, red);
    for (int it = 0; it < p.power_iters; ++it) {
      gemm<float>(D, k, T, A, 1, D, Y, 1, T, Z, 1, D, sA, sB);  // Z = Delta^T Q
      orth_cgs2(Z, D, k, coef, red);
      gemm<float>(T, k, D, A, D, 1, Z, 1, D, Y, 1, T, sA, sB);  // Y = Delta Z
      orth_cgs2(Y, T, k, coef, red);
    }
    gemm<float>(k, D, T, Y, T, 1, A, D, 1, B, D, 1, sA, sB);    // B = Q^T Delta
    for (int e = threadIdx.x; e < kp * kp; e += THREADS) C[e] = 0.f;
    __syncthreads();
    gemm<float>(k, k, D, B, D, 1, B, 1, D, C, kp, 1, sA, sB);   // C = B B^T
    jacobi_eig(C, W, kp, rot, red);
    // order the eigenpairs by decreasing eigenvalue (ties by index)
    for (int i = threadIdx.x; i < kp; i += THREADS) {
      const float li = C[i * kp + i];
      int r = 0;
      for (int j = 0; j < kp; ++j) {
        const float lj = C[j * kp + j];
        r += (lj > li) || (lj == li && j < i);
      }
      perm[r] = i;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kp * m; e += THREADS) {
      const int i = e / m, r = e % m;
      Ws[e] = W[i * kp + perm[r]];
    }
    __syncthreads();
    uint16_t* uo = p.u_out + (int64_t)s * p.out_stride;
    uint16_t* vo = p.v_out + (int64_t)s * p.out_stride;
    gemm<uint16_t>(T, m, kp, Y, 1, T, Ws, m, 1, uo, m, 1, sA, sB);  // U_m = Q W_m
    gemm<uint16_t>(D, m, kp, B, 1, D, Ws, m, 1, vo, m, 1, sA, sB);  // V_m = B^T W_m
  }
}

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

__host__ __device__ constexpr uint32_t factor_smem_bytes() {
  return (uint32_t)sizeof(float) * (2 * GT * GK + 2 * KMAX * KMAX + KMAX * 64 + KMAX + 2 * KMAX + 32) +
         (uint32_t)sizeof(int) * KMAX;
}

}  // namespace factor
}  // namespace kamera
