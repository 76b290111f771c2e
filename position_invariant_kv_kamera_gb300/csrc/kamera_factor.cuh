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
// Algorithms 4.4 and 5.1):
//   Y = Delta Omega (Omega [D][k] Gaussian, k = m + oversampling, an input);
//   Q = orth(Y);  q times: Z = orth(Delta^T Q), Q = orth(Delta Z);
//   B = Q^T Delta  [k][D];  C = B B^T = W Lambda W^T (cyclic Jacobi);
//   U_m = Q W_m (orthonormal columns),  V_m = B^T W_m (carries Sigma).
// The four products with Delta and the two output products run on tensor
// cores (tf32 operands, fp32 accumulation): in the aligned instance as
// tcgen05.mma fed by TMA, with the accumulators in tensor memory; otherwise as
// warp-level MMAs fed by cp.async.  The panel products of orth() run as
// warp-level 3xTF32 MMAs (about fp32 accuracy); the rest is fp32 on the CUDA
// cores.  orth() works on blocks of
// 16 columns: each block is projected off the finished columns (again when a
// column lost more than half its norm), then orthonormalised by Cholesky QR
// (again when the factor is ill-conditioned); a column whose remainder falls
// below 1e-4 of its norm is dropped (set to zero), so deficits of rank below
// k are handled exactly.
//
// One CTA (256 threads, two per SM) per slab at a time; each CTA owns a
// workspace region (Y [k][T], Z [k][D], B [k][D], column-major panels) in
// global memory.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace kamera {
namespace factor {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

constexpr int THREADS = 256;
constexpr int KMAX = 96;   // k = m + oversampling, padded to a multiple of 16
constexpr int GT = 64;     // GEMM tile (rows and columns)
constexpr int GK = 16;     // GEMM K step
constexpr int MAX_SWEEPS = 20;

// The operands of the aligned instance's tensor-core products as TMA tensor maps,
// encoded by the host per launch, all 3-D (x contiguous, y rows, z the slab or the
// CTA) over fp32:
//   MAP_DELTA_K   Delta {D, T, n_slabs}, box {32, 128, 1}, 128-byte swizzle (A K-major)
//   MAP_DELTA_MN  Delta {D, T, n_slabs}, box {32, 32, 1}, 128-byte swizzle of 32-byte atoms (A M-major)
//   MAP_OMEGA_MN  Omega {k, D, 1}, box {32, 32, 1}, 32-byte atoms (B N-major)
//   MAP_Y_K       Y as [kp][T] per CTA {T, kp, grid}, box {32, 64, 1}, 128-byte swizzle (B K-major)
//   MAP_Z_K       Z as [kp][D] per CTA {D, kp, grid}, box {32, 64, 1}, 128-byte swizzle (B K-major)
//   MAP_Y_MN      Y {T, kp, grid}, box {32, 32, 1}, 32-byte atoms (A M-major)
//   MAP_W_MN      W_m as [kp][m] at the start of Z {m, kp, grid}, box {32, 32, 1}, 32-byte atoms (B N-major)
//   MAP_B_MN      B as [kp][D] per CTA {D, kp, grid}, box {32, 32, 1}, 32-byte atoms (A M-major)
enum FactorMap { MAP_DELTA_K, MAP_DELTA_MN, MAP_OMEGA_MN, MAP_Y_K, MAP_Z_K, MAP_Y_MN, MAP_W_MN, MAP_B_MN, N_FACTOR_MAPS };

struct FParams {
  CUtensorMap maps[N_FACTOR_MAPS];  // the aligned instance only
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

// ---- CTA-wide fp32 GEMM: C(i,j) = alpha * sum_l A(i,l) B(l,j) (+ C(i,j)) ------------------
// Element (i,l) of A is A[i*a_rs + l*a_cs], and so on.  kAK: A is contiguous
// along K (a_cs == 1), else along M (a_rs == 1); kBK: B is contiguous along K
// (b_rs == 1), else along N (b_cs == 1).  Each operand tile sits in shared
// memory in its own orientation, so that global loads are coalesced and the
// tile is written without a transposition: K-contiguous tiles as [row][20]
// (16 used), the others as [16][64].  Every shared read is 16 bytes: four K
// values of one row, or four rows / columns of one K index.  Tiles of 64x64,
// K step 16, 256 threads; thread (ty, tx) owns rows 4ty..4ty+3 and columns
// tx + 16y (K-contiguous B) or 4tx..4tx+3; the next K step is fetched into
// registers while the current one multiplies.  Out-of-range elements read as 0.
constexpr int KS = GK + 4;  // row stride of K-contiguous tiles (16-byte aligned rows)
constexpr int GP = GT + 8;  // row stride of M/N-contiguous tiles (tensor-core fragment reads free of bank conflicts)
constexpr int TILE_FLOATS = GK * GP > GT * KS ? GK * GP : GT * KS;

// fp32 -> tf32 (round to nearest, ties away), kept in a 32-bit register
__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// D += A B on a 16x8x8 tile: tf32 operands, fp32 accumulation (warp-level tensor-core MMA)
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <typename OutT, bool kAcc, bool kAK, bool kBK, bool kTC = false>
__device__ void gemm(int M, int N, int K, const float* A, int64_t a_rs, int64_t a_cs, const float* B, int64_t b_rs,
                     int64_t b_cs, OutT* C, int64_t c_rs, int64_t c_cs, float* sA, float* sB, float alpha = 1.f) {
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  // tensor-core layout: warp w owns rows 32*(w&1) .. +31 and columns 16*(w>>1) .. +15 of the tile
  const int lane = tid & 31, warp = tid >> 5;
  const int wm = 32 * (warp & 1), wn = 16 * (warp >> 1);
  const int g = lane >> 2, t4 = lane & 3;
  constexpr int PER = GK * GT / THREADS;  // 4 elements of each operand per thread and K step
  for (int i0 = 0; i0 < M; i0 += GT) {
    for (int j0 = 0; j0 < N; j0 += GT) {
      float acc[4][4];  // SIMT: [row][column]; tensor cores: [m16 tile * 2 + n8 tile][fragment element]
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
      float ra[PER], rb[PER];
      auto fetch = [&](int l0) {
#pragma unroll
        for (int r = 0; r < PER; ++r) {
          const int e = tid + r * THREADS;
          const int i = kAK ? e / GK : e % GT, l = kAK ? e % GK : e / GT;
          const int gi = i0 + i, gl = l0 + l;
          ra[r] = (gi < M && gl < K) ? A[gi * a_rs + gl * a_cs] : 0.f;
          if (kTC) ra[r] = to_tf32(ra[r]);
          const int j = kBK ? e / GK : e % GT, l2 = kBK ? e % GK : e / GT;
          const int gj = j0 + j, gl2 = l0 + l2;
          rb[r] = (gj < N && gl2 < K) ? B[gl2 * b_rs + gj * b_cs] : 0.f;
          if (kTC) rb[r] = to_tf32(rb[r]);
        }
      };
      auto stash = [&]() {
#pragma unroll
        for (int r = 0; r < PER; ++r) {
          const int e = tid + r * THREADS;
          if (kAK) sA[(e / GK) * KS + e % GK] = ra[r];
          else sA[(e / GT) * GP + e % GT] = ra[r];
          if (kBK) sB[(e / GK) * KS + e % GK] = rb[r];
          else sB[(e / GT) * GP + e % GT] = rb[r];
        }
      };
      fetch(0);
      stash();
      __syncthreads();
      for (int l0 = 0; l0 < K; l0 += GK) {
        const bool more = l0 + GK < K;
        if (more) fetch(l0 + GK);
        if (kTC) {
          // element (i, l) of the A tile and (l, j) of the B tile, in their shared layouts
          auto at = [&](int i, int l) { return __float_as_uint(kAK ? sA[i * KS + l] : sA[l * GP + i]); };
          auto bt = [&](int l, int j) { return __float_as_uint(kBK ? sB[j * KS + l] : sB[l * GP + j]); };
#pragma unroll
          for (int k8 = 0; k8 < GK; k8 += 8) {
            uint32_t af[2][4], bf[2][2];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const int r0 = wm + 16 * mt + g;
              af[mt][0] = at(r0, k8 + t4);
              af[mt][1] = at(r0 + 8, k8 + t4);
              af[mt][2] = at(r0, k8 + t4 + 4);
              af[mt][3] = at(r0 + 8, k8 + t4 + 4);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              const int c0 = wn + 8 * nt + g;
              bf[nt][0] = bt(k8 + t4, c0);
              bf[nt][1] = bt(k8 + t4 + 4, c0);
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) mma_tf32(acc[2 * mt + nt], af[mt], bf[nt]);
          }
        }
#pragma unroll
        for (int l4 = 0; l4 < (kTC ? 0 : GK); l4 += 4) {
          float a[4][4], b[4][4];  // [row or column][k]
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            if (kAK) {
              const float4 v = *reinterpret_cast<const float4*>(sA + (ty * 4 + x) * KS + l4);
              a[x][0] = v.x; a[x][1] = v.y; a[x][2] = v.z; a[x][3] = v.w;
            } else {
              const float4 v = *reinterpret_cast<const float4*>(sA + (l4 + x) * GP + ty * 4);
              a[0][x] = v.x; a[1][x] = v.y; a[2][x] = v.z; a[3][x] = v.w;
            }
            if (kBK) {
              const float4 v = *reinterpret_cast<const float4*>(sB + (tx + 16 * x) * KS + l4);
              b[x][0] = v.x; b[x][1] = v.y; b[x][2] = v.z; b[x][3] = v.w;
            } else {
              const float4 v = *reinterpret_cast<const float4*>(sB + (l4 + x) * GP + tx * 4);
              b[0][x] = v.x; b[1][x] = v.y; b[2][x] = v.z; b[3][x] = v.w;
            }
          }
#pragma unroll
          for (int l = 0; l < 4; ++l)
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
              for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x][l], b[y][l], acc[x][y]);
        }
        __syncthreads();
        if (more) {
          stash();
          __syncthreads();
        }
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          // SIMT: row ty*4+x, column tx+16y / 4tx+y.  Tensor cores: fragment element y of
          // (m16 tile x>>1, n8 tile x&1): row g (+8 for y >= 2), column 2*t4 + (y & 1)
          const int gi = kTC ? i0 + wm + 16 * (x >> 1) + g + 8 * (y >> 1) : i0 + ty * 4 + x;
          const int gj = kTC ? j0 + wn + 8 * (x & 1) + 2 * t4 + (y & 1) : j0 + (kBK ? tx + 16 * y : tx * 4 + y);
          if (gi < M && gj < N) {
            float v = alpha * acc[x][y];
            if constexpr (kAcc) v += C[gi * c_rs + gj * c_cs];
            if constexpr (sizeof(OutT) == 2) {
              __nv_bfloat16 h = __float2bfloat16_rn(v);
              C[gi * c_rs + gj * c_cs] = *reinterpret_cast<uint16_t*>(&h);
            } else {
              C[gi * c_rs + gj * c_cs] = v;
            }
          }
        }
    }
  }
  __syncthreads();
}

// ---- tensor-core GEMM with a cp.async ring ---------------------------------------------------
// C = alpha * A B with tf32 operands and fp32 accumulation, the operand tiles
// streamed through TC_STAGES shared-memory stages by 16-byte cp.async copies
// (zero-filled past the edges).  kAK: A(i,l) = A[i*a_ld + l], else A[i + l*a_ld];
// kBK: B(l,j) = B[l + j*b_ld], else B[l*b_ld + j].  Requires 16-byte aligned
// operand bases, leading dimensions that are multiples of 4, and M, N, K
// multiples of 4 (a 16-byte chunk never straddles an edge).  Warp layout and
// fragments as in gemm<..., kTC = true>.
constexpr int TC_STAGES = 4;
constexpr int TK = 32;                                // K per stage of the tensor-core GEMM
constexpr int TKS = TK + 4;                           // row stride of its K-contiguous tiles
constexpr int TC_TILE = GT * TKS > TK * GP ? GT * TKS : TK * GP;  // floats per operand tile

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// the same with an L2 eviction policy (createpolicy)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src), "r"(src_bytes),
               "l"(policy)
               : "memory");
}
// Delta streams through L2 once per product (no slab fits alongside the others), so
// its lines go first and the CTAs' panels (Y, Z, B) stay resident between the steps
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// kStreamA / kStreamB: that operand is Delta (loaded with the evict-first policy).
template <typename OutT, bool kAK, bool kBK, bool kStreamA, bool kStreamB>
__device__ void gemm_tc(int M, int N, int K, const float* A, int64_t a_ld, const float* B, int64_t b_ld, OutT* C,
                        int64_t c_rs, int64_t c_cs, float* ring, float alpha = 1.f) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t pol = evict_first_policy();
  const int wm = 32 * (warp & 1), wn = 16 * (warp >> 1);
  const int g = lane >> 2, t4 = lane & 3;
  const int nsteps = (K + TK - 1) / TK;
  for (int i0 = 0; i0 < M; i0 += GT) {
    for (int j0 = 0; j0 < N; j0 += GT) {
      // two 16-byte chunks of each operand tile per thread and stage
      auto load_stage = [&](int slot, int l0) {
        float* sA = ring + (2 * slot) * TC_TILE;
        float* sB = sA + TC_TILE;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = tid + THREADS * h;  // chunk 0 .. 511
          int i, l, soff;
          if (kAK) { i = c >> 3; l = 4 * (c & 7); soff = i * TKS + l; }
          else     { l = c >> 4; i = 4 * (c & 15); soff = l * GP + i; }
          bool ok = i0 + i < M && l0 + l < K;
          const float* src =
              ok ? (kAK ? A + (int64_t)(i0 + i) * a_ld + l0 + l : A + (i0 + i) + (int64_t)(l0 + l) * a_ld) : A;
          if (kStreamA)
            cp_async16(smem_u32(sA + soff), src, ok ? 16u : 0u, pol);
          else
            cp_async16(smem_u32(sA + soff), src, ok ? 16u : 0u);
          int j;
          if (kBK) { j = c >> 3; l = 4 * (c & 7); soff = j * TKS + l; }
          else     { l = c >> 4; j = 4 * (c & 15); soff = l * GP + j; }
          ok = j0 + j < N && l0 + l < K;
          src = ok ? (kBK ? B + (int64_t)(j0 + j) * b_ld + l0 + l : B + (int64_t)(l0 + l) * b_ld + j0 + j) : B;
          if (kStreamB)
            cp_async16(smem_u32(sB + soff), src, ok ? 16u : 0u, pol);
          else
            cp_async16(smem_u32(sB + soff), src, ok ? 16u : 0u);
        }
      };
      float acc[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll
      for (int st = 0; st < TC_STAGES - 1; ++st) {
        if (st < nsteps) load_stage(st, st * TK);
        cp_async_commit();
      }
      for (int st = 0; st < nsteps; ++st) {
        cp_async_wait<TC_STAGES - 2>();
        __syncthreads();  // stage st landed for every thread; stage st-1 is no longer read
        const int nx = st + TC_STAGES - 1;
        if (nx < nsteps) load_stage(nx % TC_STAGES, nx * TK);
        cp_async_commit();
        const float* sA = ring + (2 * (st % TC_STAGES)) * TC_TILE;
        const float* sB = sA + TC_TILE;
        // the tf32 MMA reads the upper 19 bits of each fp32 operand; adding half a
        // tf32 ulp (bit 12) first rounds the magnitude to nearest, ties away, in
        // one integer add instead of a conversion
        auto at = [&](int i, int l) { return __float_as_uint(kAK ? sA[i * TKS + l] : sA[l * GP + i]) + 0x1000u; };
        auto bt = [&](int l, int j) { return __float_as_uint(kBK ? sB[j * TKS + l] : sB[l * GP + j]) + 0x1000u; };
#pragma unroll
        for (int k8 = 0; k8 < TK; k8 += 8) {
          uint32_t af[2][4], bf[2][2];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int r0 = wm + 16 * mt + g;
            af[mt][0] = at(r0, k8 + t4);
            af[mt][1] = at(r0 + 8, k8 + t4);
            af[mt][2] = at(r0, k8 + t4 + 4);
            af[mt][3] = at(r0 + 8, k8 + t4 + 4);
          }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int c0 = wn + 8 * nt + g;
            bf[nt][0] = bt(k8 + t4, c0);
            bf[nt][1] = bt(k8 + t4 + 4, c0);
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_tf32(acc[2 * mt + nt], af[mt], bf[nt]);
        }
      }
      cp_async_wait<0>();
      __syncthreads();  // the ring is reused by the next output tile
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int gi = i0 + wm + 16 * (x >> 1) + g + 8 * (y >> 1);
          const int gj = j0 + wn + 8 * (x & 1) + 2 * t4 + (y & 1);
          if (gi < M && gj < N) {
            const float v = alpha * acc[x][y];
            if constexpr (sizeof(OutT) == 2) {
              __nv_bfloat16 h = __float2bfloat16_rn(v);
              C[gi * c_rs + gj * c_cs] = *reinterpret_cast<uint16_t*>(&h);
            } else {
              C[gi * c_rs + gj * c_cs] = v;
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

constexpr int OB = 16;  // column block of the orthonormalisation

// ---- tall-skinny primitives over panels of n rows (column j of a panel at P + j*n) ----------

// ts_tn for a <= 24: warp w takes rows p = w, w+8, w+16 of C; each lane keeps
// four panel rows in flight.
static __device__ void ts_tn24(float* C, int ldc, const float* P, int a, const float* Q, int b, int n) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp >= a) return;  // no row of C for this warp (warp-uniform)
  float acc[3][OB];
#pragma unroll
  for (int i = 0; i < 3; ++i)
#pragma unroll
    for (int q = 0; q < OB; ++q) acc[i][q] = 0.f;
#pragma unroll 4
  for (int r = lane; r < n; r += 32) {
    float qv[OB];
#pragma unroll
    for (int q = 0; q < OB; ++q) qv[q] = q < b ? Q[(int64_t)q * n + r] : 0.f;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int p = warp + 8 * i;
      if (p < a) {
        const float pv = P[(int64_t)p * n + r];
#pragma unroll
        for (int q = 0; q < OB; ++q) acc[i][q] = fmaf(pv, qv[q], acc[i][q]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int p = warp + 8 * i;
    if (p >= a) break;  // warp-uniform
#pragma unroll
    for (int q = 0; q < OB; ++q) {
      float v = acc[i][q];
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      if (lane == 0 && q < b) C[p * ldc + q] = v;
    }
  }
}

// C[p][q] = sum_r P[p][r] Q[q][r] for p < a, q < b (b <= 16), C row-major with row
// stride ldc, in chunks of 24 rows of C; the lanes of a warp split the n rows of
// the panels and the partial sums meet by shuffles.
static __device__ void ts_tn(float* C, int ldc, const float* P, int a, const float* Q, int b, int n) {
  for (int p0 = 0; p0 < a; p0 += 24) ts_tn24(C + p0 * ldc, ldc, P + (int64_t)p0 * n, min(24, a - p0), Q, b, n);
}

// X[q][r] -= sum_{p < a} P[p][r] C[p][q] for q < b: rows r and r + THREADS per
// thread, so that each coefficient read from shared memory serves two rows.
static __device__ void ts_update(float* X, int b, const float* P, int a, const float* C, int ldc, int n) {
  for (int r = threadIdx.x; r < n; r += 2 * THREADS) {
    const int r2 = r + THREADS;
    const bool two = r2 < n;
    float x[OB], y[OB];
#pragma unroll
    for (int q = 0; q < OB; ++q) {
      x[q] = q < b ? X[(int64_t)q * n + r] : 0.f;
      y[q] = q < b && two ? X[(int64_t)q * n + r2] : 0.f;
    }
#pragma unroll 4
    for (int p = 0; p < a; ++p) {
      const float pv = P[(int64_t)p * n + r];
      const float pw = two ? P[(int64_t)p * n + r2] : 0.f;
#pragma unroll
      for (int q = 0; q < OB; ++q) {
        const float c = C[p * ldc + q];
        x[q] = fmaf(-pv, c, x[q]);
        y[q] = fmaf(-pw, c, y[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < OB; ++q)
      if (q < b) {
        X[(int64_t)q * n + r] = x[q];
        if (two) X[(int64_t)q * n + r2] = y[q];
      }
  }
}

// Cholesky G = R^T R of a b x b Gram matrix (b <= 16, row stride OB) by one warp,
// right-looking: lane c keeps column c of the partly eliminated matrix in registers
// and row j of R reaches the other lanes by shuffles.  Column j is dropped (row j
// of R zero, inv_diag[j] = 0) when its pivot -- the squared norm of what remains
// of column j after the columns before it -- is at most thr[j].  cond receives the
// ratio of the largest to the smallest kept pivot.
static __device__ void chol_drop(const float* G, float* R, float* inv_diag, const float* thr, int b, float* cond) {
  const int lane = threadIdx.x & 31;
  float col[OB];
#pragma unroll
  for (int i = 0; i < OB; ++i) col[i] = (lane < b && i < b) ? G[i * OB + lane] : 0.f;
  float rmax = 0.f, rmin = INFINITY;
#pragma unroll
  for (int j = 0; j < OB; ++j) {
    if (j >= b) break;  // warp-uniform
    const float d = __shfl_sync(0xFFFFFFFFu, col[j], j);
    const bool keep = d > thr[j];
    const float rjj = keep ? sqrtf(d) : 0.f;
    const float r = (keep && lane >= j) ? (lane == j ? rjj : col[j] / rjj) : 0.f;  // R(j, lane)
    if (lane < b) R[j * OB + lane] = r;
    if (lane == 0) inv_diag[j] = keep ? 1.f / rjj : 0.f;
    if (keep) {
      rmax = fmaxf(rmax, rjj);
      rmin = fminf(rmin, rjj);
    }
#pragma unroll
    for (int i = j + 1; i < OB; ++i) col[i] = fmaf(-__shfl_sync(0xFFFFFFFFu, r, i), r, col[i]);
  }
  __syncwarp();
  if (lane == 0) *cond = rmax > 0.f ? rmax / rmin : 1.f;
}

// X <- X R^{-1} row by row (forward substitution), R upper triangular, dropped
// columns become zero; rows r and r + THREADS per thread, so that each entry of
// R read from shared memory serves two rows.
static __device__ void ts_trsm(float* X, int b, const float* R, const float* inv_diag, int n) {
  for (int r = threadIdx.x; r < n; r += 2 * THREADS) {
    const int r2 = r + THREADS;
    const bool two = r2 < n;
    float x[OB], y[OB];
#pragma unroll
    for (int q = 0; q < OB; ++q) {
      x[q] = q < b ? X[(int64_t)q * n + r] : 0.f;
      y[q] = q < b && two ? X[(int64_t)q * n + r2] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < OB; ++j) {
      float v = x[j], w = y[j];
#pragma unroll
      for (int l = 0; l < j; ++l) {
        const float rl = R[l * OB + j];
        v = fmaf(-x[l], rl, v);
        w = fmaf(-y[l], rl, w);
      }
      const float d = inv_diag[j < b ? j : 0] * (j < b ? 1.f : 0.f);
      x[j] = v * d;
      y[j] = w * d;
    }
#pragma unroll
    for (int q = 0; q < OB; ++q)
      if (q < b) {
        X[(int64_t)q * n + r] = x[q];
        if (two) X[(int64_t)q * n + r2] = y[q];
      }
  }
}

// ---- tall-skinny primitives on the tensor cores (3xTF32) -------------------------------------
// x = hi + lo with hi = x rounded to tf32 (half an ulp added to the bits, the low 13
// cleared) and lo = x - hi (exact in fp32), rounded to tf32 the same way when the MMA
// reads it.  A product a b is taken as lo_a hi_b + hi_a lo_b + hi_a hi_b: only
// lo_a lo_b and the rounding of the lo parts are lost (below 2^-21 of |a b|), so the
// sums keep close to fp32 accuracy -- enough for the drop rule at 1e-8 of a squared
// norm -- at tensor-core speed.
__device__ __forceinline__ void split3(float x, uint32_t& hi, uint32_t& lo) {
  const uint32_t h = (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
  hi = h;
  lo = __float_as_uint(x - __uint_as_float(h)) + 0x1000u;
}

__device__ __forceinline__ void mma3(float* d, const uint32_t* ah, const uint32_t* al, const uint32_t* bh,
                                     const uint32_t* bl) {
  mma_tf32(d, al, bh);
  mma_tf32(d, ah, bl);
  mma_tf32(d, ah, bh);
}

__device__ __forceinline__ float4 ld4_or0(const float* p, bool ok) {
  return ok ? *reinterpret_cast<const float4*>(p) : make_float4(0.f, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ float f4_at(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

constexpr int TN_P = 48;  // columns of P per pass of tn_mma

// C[p][q] = sum_r P(r, p) Q(r, q) for p < a, q < b (b <= 16): P and Q column-major
// panels of n rows (column j at P + j*n; n a multiple of 4, columns 16-byte
// aligned), C row-major with row stride ldc.  Rows go to the warps in chunks of 16;
// in a chunk lane (g, t4) loads rows 4t4 .. 4t4+3 of each of its columns as one
// float4, and the chunk's two MMA K steps s = 0, 1 give K indexes t4 and t4 + 4 to
// rows 4t4 + 2s and 4t4 + 2s + 1 (a permutation of the rows, which the sum does not
// see).  The warps' partial sums meet in scr (8 x TN_P x 16 floats of shared
// memory) and are added in warp order.
static __device__ void tn_mma(float* C, int ldc, const float* P, int a, const float* Q, int b, int n, float* scr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
  const int nch = (n + 15) >> 4;
  for (int p0 = 0; p0 < a; p0 += TN_P) {
    const int ap = min(TN_P, a - p0);
    float acc[3][2][4];
#pragma unroll
    for (int mt = 0; mt < 3; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll 1
    for (int ch = warp; ch < nch; ch += 8) {
      const int r = 16 * ch + 4 * t4;
      const bool rok = r < n;  // n % 4 == 0: a float4 is wholly inside or wholly outside
      float4 pv[3][2], qv[2];
#pragma unroll
      for (int mt = 0; mt < 3; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = p0 + 16 * mt + 8 * h + g;
          pv[mt][h] = ld4_or0(P + (int64_t)c * n + r, rok && 16 * mt < ap && c < a);
        }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 8 * nt + g;
        qv[nt] = ld4_or0(Q + (int64_t)c * n + r, rok && c < b);
      }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        uint32_t bh[2][2], bl[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          split3(f4_at(qv[nt], 2 * s2), bh[nt][0], bl[nt][0]);
          split3(f4_at(qv[nt], 2 * s2 + 1), bh[nt][1], bl[nt][1]);
        }
#pragma unroll
        for (int mt = 0; mt < 3; ++mt) {
          if (16 * mt >= ap) break;  // warp-uniform
          uint32_t ah[4], al[4];
          split3(f4_at(pv[mt][0], 2 * s2), ah[0], al[0]);      // (g, t4)
          split3(f4_at(pv[mt][1], 2 * s2), ah[1], al[1]);      // (g + 8, t4)
          split3(f4_at(pv[mt][0], 2 * s2 + 1), ah[2], al[2]);  // (g, t4 + 4)
          split3(f4_at(pv[mt][1], 2 * s2 + 1), ah[3], al[3]);  // (g + 8, t4 + 4)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            if (8 * nt < b) mma3(acc[mt][nt], ah, al, bh[nt], bl[nt]);
        }
      }
    }
    float* sw = scr + warp * (TN_P * OB);
#pragma unroll
    for (int mt = 0; mt < 3; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sw[(16 * mt + g + 8 * (e >> 1)) * OB + 8 * nt + 2 * t4 + (e & 1)] = acc[mt][nt][e];
    __syncthreads();
    for (int e = threadIdx.x; e < ap * OB; e += THREADS) {
      const int pp = e / OB, q = e % OB;
      if (q < b) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < THREADS / 32; ++w) sum += scr[w * (TN_P * OB) + e];
        C[(p0 + pp) * ldc + q] = sum;
      }
    }
    __syncthreads();
  }
}

// Orthonormalise the k columns (length n, column j at X + j*n) in place, one
// block of 16 columns at a time: the block is projected off the finished
// columns (classical block Gram-Schmidt), a second time when a column lost
// more than half of its squared norm in the first projection ("twice is
// enough", Giraud, Langou & Rozloznik 2005), then orthonormalised by Cholesky
// QR (Gram matrix, Cholesky, triangular solve), a second time when the first
// Cholesky factor is ill-conditioned (largest / smallest pivot above 16).  A
// column whose remainder falls below 1e-4 of its original norm is dependent
// and becomes zero (its Cholesky pivot is dropped).  One pass over the first
// J0 + 16 columns gives both the first projection coefficients and the block's
// original Gram matrix.  kTC: the coefficient and Gram products on the tensor
// cores (3xTF32; n a multiple of 4, columns 16-byte aligned), else the fp32
// warp primitives; the projection update and the triangular solve are fp32
// loops over rows, two rows per thread, either way (they keep more loads in
// flight than a warp tile of MMAs does, and each shared-memory coefficient
// read serves both rows).
// Scratch (shared): cblk [kp][OB] (coefficients above row J0, the block's Gram
// matrix from row J0), rmat [OB][OB], inv_diag [OB], thr [OB], orig [OB]
// (squared original norms), cond [1]; scr 8*TN_P*OB floats (kTC).
template <bool kTC>
__device__ void orth_block(float* X, int n, int k, float* cblk, float* rmat, float* inv_diag, float* thr, float* scr) {
  float* orig = thr + OB;
  float* cond = orig + OB;
  auto tn = [&](float* C, const float* P, int a, const float* Q, int b) {
    if constexpr (kTC)
      tn_mma(C, OB, P, a, Q, b, n, scr);
    else
      ts_tn(C, OB, P, a, Q, b, n);
  };
  for (int J0 = 0; J0 < k; J0 += OB) {
    const int b = min(OB, k - J0);
    float* XJ = X + (int64_t)J0 * n;
    float* gram = cblk + J0 * OB;
    tn(cblk, X, J0 + b, XJ, b);  // [Q_< | X_J]^T X_J
    __syncthreads();
    if (threadIdx.x < b) {  // squared original norms -> drop thresholds (1e-4 of the norm)
      orig[threadIdx.x] = gram[threadIdx.x * OB + threadIdx.x];
      thr[threadIdx.x] = 1e-8f * orig[threadIdx.x];
    }
    __syncthreads();
    bool fresh_gram = true;  // gram holds the Gram matrix of the current X_J
    for (int pass = 0; pass < 2 && J0 > 0; ++pass) {
      if (pass == 1) {
        tn(cblk, X, J0, XJ, b);  // cblk [J0][b] = Q_<^T X_J
        __syncthreads();
      }
      ts_update(XJ, b, X, J0, cblk, OB, n);  // X_J -= Q_< cblk
      __syncthreads();
      tn(gram, XJ, b, XJ, b);
      __syncthreads();
      bool again = false;
      for (int j = 0; j < b; ++j) again |= gram[j * OB + j] < 0.5f * orig[j];
      if (!again) break;  // block-uniform: every thread reads the same shared values
      __syncthreads();    // the next pass rewrites cblk and gram
    }
    for (int pass = 0; pass < 2; ++pass) {
      if (!fresh_gram) {
        tn(gram, XJ, b, XJ, b);
        __syncthreads();
      }
      if (threadIdx.x < 32) {
        if (pass == 1 && threadIdx.x < b) thr[threadIdx.x] = 1e-8f * gram[threadIdx.x * OB + threadIdx.x];
        __syncwarp();
        chol_drop(gram, rmat, inv_diag, thr, b, cond);
      }
      __syncthreads();
      ts_trsm(XJ, b, rmat, inv_diag, n);
      const bool again = *cond > 16.f;
      __syncthreads();
      fresh_gram = false;
      if (!again) break;
    }
  }
}

// Cyclic Jacobi eigen-decomposition of the symmetric kp x kp matrix C (row
// major, in shared memory) with the parallel (round-robin tournament) order:
// each round rotates kp/2 disjoint planes at once.  On return the diagonal of
// C holds the eigenvalues and the columns of W the eigenvectors.
static __device__ void jacobi_eig(float* C, float* W, int kp, int ld, float* rot, float* red) {
  const int tid = threadIdx.x;
  for (int e = tid; e < kp * kp; e += THREADS) W[(e / kp) * ld + e % kp] = (e / kp == e % kp) ? 1.f : 0.f;
  __syncthreads();
  const int half = kp / 2;
  // (row, column) of element tid of a half-wide index space, and the step of THREADS elements
  const int e_i0 = tid / half, e_j0 = tid - e_i0 * half, e_qs = THREADS / half, e_rs = THREADS - e_qs * half;
  for (int sweep = 0; sweep < MAX_SWEEPS; ++sweep) {
    float off = 0.f, tot = 0.f;
    for (int e = tid; e < kp * kp; e += THREADS) {
      const float x = C[(e / kp) * ld + e % kp];
      tot += x * x;
      if (e / kp != e % kp) off += x * x;
    }
    off = block_sum(off, red);
    tot = block_sum(tot, red);
    if (off <= 1e-10f * tot || tot == 0.f) break;
    // pair tid of round r: players a = 1 + (tid - 1 + r) mod (kp - 1) (0 for tid 0) and
    // b = 1 + (kp - 2 - tid + r) mod (kp - 1) of the rotated ring, stepped without division
    int pa = tid == 0 ? 0 : tid, pb = kp - 1 - tid;
    for (int round = 0; round < kp - 1; ++round) {
      if (tid < half) {
        const int p = min(pa, pb), q = max(pa, pb);
        const float app = C[p * ld + p], aqq = C[q * ld + q], apq = C[p * ld + q];
        float c = 1.f, s = 0.f;
        if (apq != 0.f && fabsf(apq) > 1e-30f) {
          // the angle in fast arithmetic: a rotation that leaves a small a_pq is
          // corrected by the next sweep, and the rotation itself stays orthogonal
          const float zeta = __fdividef(aqq - app, 2.f * apq);
          const float t = copysignf(__fdividef(1.f, fabsf(zeta) + sqrtf(1.f + zeta * zeta)), zeta);
          c = rsqrtf(1.f + t * t);
          s = c * t;
        }
        *reinterpret_cast<float4*>(rot + 4 * tid) = make_float4(__int_as_float(p), __int_as_float(q), c, s);
        if (tid > 0) pa = pa == kp - 1 ? 1 : pa + 1;
        pb = pb == kp - 1 ? 1 : pb + 1;
      }
      __syncthreads();
      // The pairs are disjoint and cover every index, so C splits into 2x2 blocks
      // B_ij (rows p_i, q_i; columns p_j, q_j), each of which becomes G_i B_ij G_j^T
      // with G = [c -s; s c]; W <- W G^T on the column pairs.  One step, each
      // element read and written once.
      // Block e = i * half + j of C and pair e = jr * half + i of W for e = tid, tid +
      // THREADS, ...: every thread takes about the same share (indexes stepped
      // without division).
      for (int e = tid, i = e_i0, j = e_j0; e < half * half; e += THREADS) {
        const float4 ri = *reinterpret_cast<const float4*>(rot + 4 * i);
        const float4 rj = *reinterpret_cast<const float4*>(rot + 4 * j);
        const int pi = __float_as_int(ri.x), qi = __float_as_int(ri.y);
        const int pj = __float_as_int(rj.x), qj = __float_as_int(rj.y);
        const float b00 = C[pi * ld + pj], b01 = C[pi * ld + qj], b10 = C[qi * ld + pj], b11 = C[qi * ld + qj];
        // rows: G_i B
        const float u00 = ri.z * b00 - ri.w * b10, u01 = ri.z * b01 - ri.w * b11;
        const float u10 = ri.w * b00 + ri.z * b10, u11 = ri.w * b01 + ri.z * b11;
        // columns: (G_i B) G_j^T
        C[pi * ld + pj] = rj.z * u00 - rj.w * u01;
        C[pi * ld + qj] = rj.w * u00 + rj.z * u01;
        C[qi * ld + pj] = rj.z * u10 - rj.w * u11;
        C[qi * ld + qj] = rj.w * u10 + rj.z * u11;
        j += e_rs;
        i += e_qs;
        if (j >= half) {
          j -= half;
          ++i;
        }
      }
      for (int e = tid, jr = e_i0, i = e_j0; e < kp * half; e += THREADS) {
        const float4 ri = *reinterpret_cast<const float4*>(rot + 4 * i);
        float* w = W + jr * ld;
        const int pi = __float_as_int(ri.x), qi = __float_as_int(ri.y);
        const float xp = w[pi], xq = w[qi];
        w[pi] = ri.z * xp - ri.w * xq;
        w[qi] = ri.w * xp + ri.z * xq;
        i += e_rs;
        jr += e_qs;
        if (i >= half) {
          i -= half;
          ++jr;
        }
      }
      __syncthreads();
    }
  }
}

// ---- tall-skinny tensor-core GEMM: all of N (<= 48) in one tile ------------------------------
// C = alpha * A B for N <= TN: output tiles of TM x TN, warp w owns rows 32 (w & 3) .. +31
// and columns 24 (w >> 2) .. +23 (two m16 x three n8 fragments), so that no warp idles at
// N = 48 and the skinny operand is re-read once per 128 rows.  Operands stream through
// TALL_STAGES stages of K = TK as in gemm_tc, with its layouts, edge rules and rounding.
constexpr int TM = 128, TN = 48;
constexpr int GPA = TM + 8, GPB = TN + 8;  // row strides of M/N-contiguous tiles (conflict-free fragment reads)
constexpr int TALL_STAGES = 3;
constexpr int TALL_A = TM * TKS > TK * GPA ? TM * TKS : TK * GPA;
constexpr int TALL_B = TN * TKS > TK * GPB ? TN * TKS : TK * GPB;
constexpr int TALL_STAGE = TALL_A + TALL_B;
constexpr int RING_FLOATS =
    2 * TC_STAGES * TC_TILE > TALL_STAGES * TALL_STAGE ? 2 * TC_STAGES * TC_TILE : TALL_STAGES * TALL_STAGE;

template <typename OutT, bool kAK, bool kBK, bool kStreamA, bool kStreamB>
__device__ void gemm_tall(int M, int N, int K, const float* A, int64_t a_ld, const float* B, int64_t b_ld, OutT* C,
                          int64_t c_rs, int64_t c_cs, float* ring, float alpha = 1.f) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = 32 * (warp & 3), wn = 24 * (warp >> 2);
  const int g = lane >> 2, t4 = lane & 3;
  const uint64_t pol = evict_first_policy();
  const int nsteps = (K + TK - 1) / TK;
  for (int i0 = 0; i0 < M; i0 += TM) {
    auto load_stage = [&](int slot, int l0) {
      float* sA = ring + slot * TALL_STAGE;
      float* sB = sA + TALL_A;
#pragma unroll
      for (int h = 0; h < TM * TK / 4 / THREADS; ++h) {  // four 16-byte chunks of A per thread
        const int c = tid + THREADS * h;
        int i, l, soff;
        if (kAK) { i = c >> 3; l = 4 * (c & 7); soff = i * TKS + l; }
        else     { l = c >> 5; i = 4 * (c & 31); soff = l * GPA + i; }
        const bool ok = i0 + i < M && l0 + l < K;
        const float* src =
            ok ? (kAK ? A + (int64_t)(i0 + i) * a_ld + l0 + l : A + (i0 + i) + (int64_t)(l0 + l) * a_ld) : A;
        if (kStreamA)
          cp_async16(smem_u32(sA + soff), src, ok ? 16u : 0u, pol);
        else
          cp_async16(smem_u32(sA + soff), src, ok ? 16u : 0u);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // 384 chunks of B
        const int c = tid + THREADS * h;
        if (c < TN * TK / 4) {
          int j, l, soff;
          if (kBK) { j = c >> 3; l = 4 * (c & 7); soff = j * TKS + l; }
          else     { l = c / (TN / 4); j = 4 * (c % (TN / 4)); soff = l * GPB + j; }
          const bool ok = j < N && l0 + l < K;
          const float* src = ok ? (kBK ? B + (int64_t)j * b_ld + l0 + l : B + (int64_t)(l0 + l) * b_ld + j) : B;
          if (kStreamB)
            cp_async16(smem_u32(sB + soff), src, ok ? 16u : 0u, pol);
          else
            cp_async16(smem_u32(sB + soff), src, ok ? 16u : 0u);
        }
      }
    };
    float acc[2][3][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 3; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][b][e] = 0.f;
#pragma unroll
    for (int st = 0; st < TALL_STAGES - 1; ++st) {
      if (st < nsteps) load_stage(st, st * TK);
      cp_async_commit();
    }
    for (int st = 0; st < nsteps; ++st) {
      cp_async_wait<TALL_STAGES - 2>();
      __syncthreads();  // stage st landed for every thread; stage st-1 is no longer read
      const int nx = st + TALL_STAGES - 1;
      if (nx < nsteps) load_stage(nx % TALL_STAGES, nx * TK);
      cp_async_commit();
      const float* sA = ring + (st % TALL_STAGES) * TALL_STAGE;
      const float* sB = sA + TALL_A;
      // tf32 rounding by half an ulp added to the bits, as in gemm_tc
      auto at = [&](int i, int l) { return __float_as_uint(kAK ? sA[i * TKS + l] : sA[l * GPA + i]) + 0x1000u; };
      auto bt = [&](int l, int j) { return __float_as_uint(kBK ? sB[j * TKS + l] : sB[l * GPB + j]) + 0x1000u; };
#pragma unroll
      for (int k8 = 0; k8 < TK; k8 += 8) {
        uint32_t af[2][4], bf[3][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int r0 = wm + 16 * mt + g;
          af[mt][0] = at(r0, k8 + t4);
          af[mt][1] = at(r0 + 8, k8 + t4);
          af[mt][2] = at(r0, k8 + t4 + 4);
          af[mt][3] = at(r0 + 8, k8 + t4 + 4);
        }
#pragma unroll
        for (int nt = 0; nt < 3; ++nt) {
          const int c0 = wn + 8 * nt + g;
          bf[nt][0] = bt(k8 + t4, c0);
          bf[nt][1] = bt(k8 + t4 + 4, c0);
        }
#pragma unroll
        for (int nt = 0; nt < 3; ++nt) {
          if (wn + 8 * nt >= N) break;  // warp-uniform: columns past N are zero
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) mma_tf32(acc[mt][nt], af[mt], bf[nt]);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // the ring is reused by the next output tile
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 3; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int gi = i0 + wm + 16 * mt + g + 8 * (e >> 1);
          const int gj = wn + 8 * nt + 2 * t4 + (e & 1);
          if (gi < M && gj < N) {
            const float v = alpha * acc[mt][nt][e];
            if constexpr (sizeof(OutT) == 2) {
              __nv_bfloat16 hv = __float2bfloat16_rn(v);
              C[gi * c_rs + gj * c_cs] = *reinterpret_cast<uint16_t*>(&hv);
            } else {
              C[gi * c_rs + gj * c_cs] = v;
            }
          }
        }
  }
  __syncthreads();
}

// ---- tall-skinny products on the 5th-generation tensor cores -------------------------------
// The products of the aligned instance with N <= 64: tcgen05.mma kind::tf32 into fp32
// accumulators of 128 TMEM lanes x 64 columns (N padded to 64 with zero columns of B),
// two of them, so that the epilogue of one 128-row tile overlaps the MMAs of the next.
// The operands arrive by TMA in TC_RING_STAGES stages of 24 KB (K = 32), in the
// canonical layouts the MMA reads: a K-contiguous operand K-major (128-byte rows, the
// 128-byte swizzle), an M- or N-contiguous one MN-major (K rows of 32 values, 128
// bytes, with the 128-byte swizzle of 32-byte atomicity that tcgen05 reads for
// 32-bit MN-major operands; atoms of 32 along M or N 4096 bytes apart), so neither
// needs a transposition.  One thread issues the copies (a stage is refilled once the
// MMAs that read it committed), one issues the MMAs (four K = 8 per stage), and warps
// 4-7 move each finished accumulator to C; the stages of all the tiles of a product
// form one stream.  The tensor core takes the upper 19 bits of each fp32 word (tf32 by
// truncation): the deficits are read as they are, and every operand this kernel
// writes itself (the fp32 products' outputs, the final Q, W_m) is stored rounded to
// the nearest tf32 value, so that for those the truncation is exact.  Out-of-range
// rows and columns arrive as zeros.
constexpr int TC_RING_STAGES = 4;
constexpr int TC_N = 64;                       // accumulator columns: N <= TC_N
constexpr uint32_t TCA_BYTES = TM * TK * 4;    // A stage: 128 x 32 fp32
constexpr uint32_t TCB_BYTES = TC_N * TK * 4;  // B stage: 64 x 32 fp32
constexpr uint32_t TC_STAGE_BYTES = TCA_BYTES + TCB_BYTES;
constexpr int TC_RING_FLOATS = (TC_RING_STAGES * TC_STAGE_BYTES + 1024) / 4;  // + alignment to 1024 bytes
constexpr uint32_t TC_TMEM_COLS = 2 * TC_N;

struct TcState {  // per CTA, in shared memory
  uint64_t full[TC_RING_STAGES];   // stage landed
  uint64_t empty[TC_RING_STAGES];  // stage's MMAs completed
  uint64_t accfull[2];             // accumulator b holds a finished tile
  uint64_t accempty[2];            // accumulator b was read out (one arrival per epilogue warp)
  uint32_t tmem;
};

// Position of a CTA in its stream of tensor-core stages and tiles, across products:
// the phases of the barriers follow from it.
struct TcCursor {
  uint32_t stage = 0, tile = 0;
};

// fp32 -> the nearest tf32 value (ties away from zero), as an fp32 word whose low 13
// bits are zero: operands this kernel writes for later products are stored rounded,
// so that the tensor core's truncation leaves them unchanged.
__device__ __forceinline__ float tf32_rn(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// Bounded wait (2 s): on expiry it returns and the products are wrong, the kernel
// never hangs.
__device__ __forceinline__ void tc_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 2000000000ull) return;
}

// A 3-D TMA tile load with an L2 cache policy: the deficit streams through with
// evict-first, so that it does not push the per-CTA workspace panels out of L2.
__device__ __forceinline__ void tma_load_3d_policy(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                                   int32_t y, int32_t z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Set-up and tear-down of the accumulators and the barriers; whole CTA.
__device__ __forceinline__ void tc_setup(TcState* tc) {
  if (threadIdx.x < 32) {
    tmem_alloc(&tc->tmem, TC_TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < TC_RING_STAGES; ++i) {
      mbar_init(&tc->full[i], 1);
      mbar_init(&tc->empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tc->accfull[b], 1);
      mbar_init(&tc->accempty[b], 4);
    }
    fence_mbar_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
}

__device__ __forceinline__ void tc_teardown(TcState* tc) {
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (threadIdx.x < 32) tmem_dealloc(tc->tmem, TC_TMEM_COLS);
}

// C = A B (M x N, N <= 64) with A(i, l) and B(l, j) read through the tensor maps amap
// and bmap at slab or CTA coordinate az / bz.  kAK: A is K-contiguous (map box
// {32 along K, 128 rows}), else M-contiguous (box {32 along M, 32 K rows}, four per
// stage); kBK: B is K-contiguous (box {32 along K, 64 columns}), else N-contiguous
// (box {32 along N, 32 K rows}, two per stage).  Element (i, j) of C goes to
// C[i*c_rs + j*c_cs].  Whole CTA.
template <typename OutT, bool kAK, bool kBK>
__device__ void gemm_tall_tma(int M, int N, int K, const CUtensorMap* amap, int az, const CUtensorMap* bmap, int bz,
                              OutT* C, int64_t c_rs, int64_t c_cs, float* ring, TcState* tc, TcCursor& cur) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int R = TC_RING_STAGES;
  const uint32_t pad = ((smem_u32(ring) + 1023u) & ~1023u) - smem_u32(ring);
  unsigned char* stages = reinterpret_cast<unsigned char*>(ring) + pad;
  const int nsteps = (K + TK - 1) / TK, ntiles = (M + TM - 1) / TM, total = nsteps * ntiles;
  const uint32_t g0 = cur.stage, t0 = cur.tile;
  constexpr uint32_t IDESC = umma_idesc_tf32_f32(TM, TC_N, !kAK, !kBK);
  // the operands this CTA wrote with plain stores (earlier products, the
  // orthonormalisation), and the plain uses of the ring since the last product,
  // ordered before the TMA traffic
  fence_proxy_async_global();
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {  // copies: A (the deficit, or a panel) streams evict-first, B stays in L2
    const uint64_t pol = evict_first_policy();
    for (int idx = 0; idx < total; ++idx) {
      const uint32_t g = g0 + (uint32_t)idx, slot = g % R;
      if (g >= (uint32_t)R) tc_wait(&tc->empty[slot], ((g / R) - 1u) & 1u);
      const int tt = idx / nsteps, i0 = tt * TM, l0 = (idx - tt * nsteps) * TK;
      unsigned char* sA = stages + slot * TC_STAGE_BYTES;
      unsigned char* sB = sA + TCA_BYTES;
      uint64_t* bar = &tc->full[slot];
      mbar_arrive_expect_tx(bar, TC_STAGE_BYTES);
      if (kAK) {
        tma_load_3d_policy(sA, amap, bar, l0, i0, az, pol);
      } else {
#pragma unroll
        for (int a = 0; a < TM / 32; ++a) tma_load_3d_policy(sA + 4096 * a, amap, bar, i0 + 32 * a, l0, az, pol);
      }
      if (kBK) {
        tma_load_3d(sB, bmap, bar, l0, 0, bz);
      } else {
#pragma unroll
        for (int b = 0; b < TC_N / 32; ++b) tma_load_3d(sB + 4096 * b, bmap, bar, 32 * b, l0, bz);
      }
    }
  } else if (tid == 32) {  // MMAs
    int tt = 0, st = 0;
    for (int idx = 0; idx < total; ++idx) {
      const uint32_t g = g0 + (uint32_t)idx, slot = g % R, gt = t0 + (uint32_t)tt, acc = tc->tmem + (gt & 1u) * TC_N;
      if (st == 0 && gt >= 2u) tc_wait(&tc->accempty[gt & 1u], ((gt >> 1) - 1u) & 1u);
      tc_wait(&tc->full[slot], (g / R) & 1u);
      tc_fence_after_sync();
      const uint32_t sA = smem_u32(stages + slot * TC_STAGE_BYTES), sB = sA + TCA_BYTES;
#pragma unroll
      for (int ks = 0; ks < TK / 8; ++ks) {  // K = 8 per MMA: 32 bytes of a K-major row, two MN-major K groups
        const uint64_t ad = kAK ? umma_desc_kmajor_sw(sA + 32u * ks, 128u)
                                : umma_desc_mnmajor_sw128b32(sA + 1024u * ks, 4096u, 512u);
        const uint64_t bd = kBK ? umma_desc_kmajor_sw(sB + 32u * ks, 128u)
                                : umma_desc_mnmajor_sw128b32(sB + 1024u * ks, 4096u, 512u);
        umma_tf32(acc, ad, bd, IDESC, (st > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(&tc->empty[slot]);
      if (st == nsteps - 1) umma_commit(&tc->accfull[gt & 1u]);
      if (++st == nsteps) {
        st = 0;
        ++tt;
      }
    }
  } else if (warp >= 4) {  // epilogue: warp w reads TMEM lanes 32 (w - 4) .. +31, its rows of the tile
    const int q = warp - 4;
    for (int tt = 0; tt < ntiles; ++tt) {
      const uint32_t gt = t0 + (uint32_t)tt;
      tc_wait(&tc->accfull[gt & 1u], (gt >> 1) & 1u);
      __syncwarp();
      tc_fence_after_sync();
      const int gi = tt * TM + 32 * q + lane;
      for (int cb = 0; cb < N; cb += 32) {
        uint32_t v[32];
        tmem_ld32(tc->tmem + ((uint32_t)(32 * q) << 16) + (gt & 1u) * TC_N + (uint32_t)cb, v);
        tmem_ld_wait();
        if (gi < M) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (cb + j < N) {
              const float x = __uint_as_float(v[j]);
              if constexpr (sizeof(OutT) == 2) {
                __nv_bfloat16 hv = __float2bfloat16_rn(x);
                C[gi * c_rs + (cb + j) * c_cs] = *reinterpret_cast<uint16_t*>(&hv);
              } else {
                C[gi * c_rs + (cb + j) * c_cs] = tf32_rn(x);  // an operand of a later product
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tc->accempty[gt & 1u]);
    }
  }
  cur.stage = g0 + (uint32_t)total;
  cur.tile = t0 + (uint32_t)ntiles;
  __syncthreads();  // C is written; the ring is free for the caller once its MMAs completed (seen above)
}

// Shared memory of one CTA, in floats, for a given kp and m.  The first region holds
// the GEMM stages while the Delta products, the orthonormalisations and the output
// products run, and C, W and Ws (the eigenproblem) at its end while they do not; the
// fp32 GEMM tiles at its start serve the products with C alive.
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int eig_floats(int kp, int m) { return 2 * kp * (kp + 1) + kp * m; }
__host__ __device__ constexpr int region_floats(int kp, int m) {
  return cmax(cmax(RING_FLOATS, TC_RING_FLOATS), 2 * TILE_FLOATS + eig_floats(kp, m));
}
__host__ __device__ constexpr int factor_smem_floats(int kp, int m) {
  return region_floats(kp, m) + kp * OB + 2 * kp + 32 + kp + OB * OB + 3 * OB + 4;
}

// kAligned: T, D, k and the slab stride are multiples of 4 and Delta, Omega and the
// workspace are 16-byte aligned (the host checks it), so every product takes the
// tensor-core path and the fp32 fallbacks are not compiled in -- they would set the
// register budget of the whole kernel.
template <bool kAligned>
__global__ void __launch_bounds__(THREADS, 2) factor_kernel(const __grid_constant__ FParams p) {
  extern __shared__ __align__(16) float fsm[];
  const int T = p.T, D = p.D, k = p.k, kp = p.kp, m = p.m;
  float* ring = fsm;                  // the tensor-core GEMMs' stages
  float* sA = ring;                   // the first two fp32-GEMM tiles overlay the ring
  float* sB = sA + TILE_FLOATS;
  const int region = region_floats(kp, m);
  float* C = ring + region - eig_floats(kp, m);  // kp*(kp+1), past the fp32 tiles
  const int ld = kp + 1;              // row stride of C and W: rows fall on different banks
  float* W = C + kp * ld;             // kp*ld
  float* Ws = W + kp * ld;            // kp*m: sorted leading eigenvectors
  float* cblk = ring + region;        // kp*OB: projection coefficients of a column block
  float* rot = cblk + kp * OB;        // 2*kp
  float* red = rot + 2 * kp;          // 32
  int* perm = reinterpret_cast<int*>(red + 32);  // kp
  float* rmat = red + 32 + kp;        // OB*OB
  float* inv_diag = rmat + OB * OB;   // OB
  float* thr = inv_diag + OB;         // OB, then orig (OB) and cond (1) for orth_block

  float* Y = p.work + blockIdx.x * p.work_per_cta;  // [kp][T] column-major
  float* Z = Y + (int64_t)kp * T;                   // [kp][D]
  float* B = Z + (int64_t)kp * D;                   // [kp][D]: row i of B contiguous

  // rows k..kp-1 of B are never written: keep them zero for the V_m product
  for (int64_t e = (int64_t)k * D + threadIdx.x; e < (int64_t)kp * D; e += THREADS) B[e] = 0.f;
  // the cp.async path needs 16-byte chunks that never straddle an edge
  const bool ring_ok = kAligned || (((T | D | k) & 3) == 0 && (p.delta_stride & 3) == 0 &&
                                    ((reinterpret_cast<uintptr_t>(p.delta) | reinterpret_cast<uintptr_t>(p.omega)) &
                                     15u) == 0);
  // the tensor-core panel primitives need 16-byte aligned panel columns
  const bool panel_ok = kAligned || (((T | D) & 3) == 0 && (reinterpret_cast<uintptr_t>(p.work) & 15u) == 0);
  // every product in one column tile: up to 64 columns on tcgen05, 48 on mma.sync
  const bool tall = ring_ok && kp <= (kAligned ? TC_N : TN);
  __shared__ TcState tcs;  // the aligned instance's accumulator and stage barriers
  TcCursor tcur;           // this CTA's tensor-core stages and tiles so far (the barriers' phases)
  if (kAligned && tall) tc_setup(&tcs);
  auto orth = [&](float* X, int n) {
    if (panel_ok)
      orth_block<true>(X, n, k, cblk, rmat, inv_diag, thr, ring);
    else
      orth_block<false>(X, n, k, cblk, rmat, inv_diag, thr, ring);
  };
  for (int s = blockIdx.x; s < p.n_slabs; s += gridDim.x) {
    const float* A = p.delta + (int64_t)s * p.delta_stride;  // [T][D]
    // Y = Delta Omega (columns k..kp-1 stay zero)
    for (int64_t e = threadIdx.x; e < (int64_t)kp * T; e += THREADS) Y[e] = 0.f;
    __syncthreads();
    if (tall) {
      if constexpr (kAligned)
        gemm_tall_tma<float, true, false>(T, k, D, &p.maps[MAP_DELTA_K], s, &p.maps[MAP_OMEGA_MN], 0, Y, 1, T, ring,
                                          &tcs, tcur);
      else
        gemm_tall<float, true, false, true, false>(T, k, D, A, D, p.omega, k, Y, 1, T, ring);
    } else if (ring_ok)
      gemm_tc<float, true, false, true, false>(T, k, D, A, D, p.omega, k, Y, 1, T, ring);
    else
      gemm<float, false, true, false, true>(T, k, D, A, D, 1, p.omega, k, 1, Y, 1, T, sA, sB);
    orth(Y, T);
    for (int it = 0; it < p.power_iters; ++it) {
      if (tall) {  // Z = Delta^T Q
        if constexpr (kAligned)
          gemm_tall_tma<float, false, true>(D, k, T, &p.maps[MAP_DELTA_MN], s, &p.maps[MAP_Y_K], blockIdx.x, Z, 1, D,
                                            ring, &tcs, tcur);
        else
          gemm_tall<float, false, true, true, false>(D, k, T, A, D, Y, T, Z, 1, D, ring);
      } else if (ring_ok)
        gemm_tc<float, false, true, true, false>(D, k, T, A, D, Y, T, Z, 1, D, ring);
      else
        gemm<float, false, false, true, true>(D, k, T, A, 1, D, Y, 1, T, Z, 1, D, sA, sB);
      orth(Z, D);
      if (tall) {  // Y = Delta Z
        if constexpr (kAligned)
          gemm_tall_tma<float, true, true>(T, k, D, &p.maps[MAP_DELTA_K], s, &p.maps[MAP_Z_K], blockIdx.x, Y, 1, T,
                                           ring, &tcs, tcur);
        else
          gemm_tall<float, true, true, true, false>(T, k, D, A, D, Z, D, Y, 1, T, ring);
      } else if (ring_ok)
        gemm_tc<float, true, true, true, false>(T, k, D, A, D, Z, D, Y, 1, T, ring);
      else
        gemm<float, false, true, true, true>(T, k, D, A, D, 1, Z, 1, D, Y, 1, T, sA, sB);
      orth(Y, T);
    }
    if constexpr (kAligned) {  // the final Q, an operand of B = Q^T Delta and U_m = Q W_m: rounded to tf32
      if (tall) {  // k * T is a multiple of 4 and Y 16-byte aligned here
        float4* y4 = reinterpret_cast<float4*>(Y);
#pragma unroll 4
        for (int64_t e = threadIdx.x; e < (int64_t)k * T / 4; e += THREADS) {
          float4 v = y4[e];
          v.x = tf32_rn(v.x);
          v.y = tf32_rn(v.y);
          v.z = tf32_rn(v.z);
          v.w = tf32_rn(v.w);
          y4[e] = v;
        }
        __syncthreads();
      }
    }
    if (tall) {  // B = Q^T Delta, formed as B^T = Delta^T Q (D x k, column j = row j of B)
      if constexpr (kAligned)
        gemm_tall_tma<float, false, true>(D, k, T, &p.maps[MAP_DELTA_MN], s, &p.maps[MAP_Y_K], blockIdx.x, B, 1, D,
                                          ring, &tcs, tcur);
      else
        gemm_tall<float, false, true, true, false>(D, k, T, A, D, Y, T, B, 1, D, ring);
    } else if (ring_ok)  // B = Q^T Delta
      gemm_tc<float, true, false, false, true>(k, D, T, Y, T, A, D, B, D, 1, ring);
    else
      gemm<float, false, true, false, true>(k, D, T, Y, T, 1, A, D, 1, B, D, 1, sA, sB);
    for (int e = threadIdx.x; e < kp * ld; e += THREADS) C[e] = 0.f;
    __syncthreads();
    gemm<float, false, true, true>(k, k, D, B, D, 1, B, 1, D, C, ld, 1, sA, sB);   // C = B B^T
    jacobi_eig(C, W, kp, ld, rot, red);
    // order the eigenpairs by decreasing eigenvalue (ties by index)
    for (int i = threadIdx.x; i < kp; i += THREADS) {
      const float li = C[i * ld + i];
      int r = 0;
      for (int j = 0; j < kp; ++j) {
        const float lj = C[j * ld + j];
        r += (lj > li) || (lj == li && j < i);
      }
      perm[r] = i;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kp * m; e += THREADS) {
      const int i = e / m, r = e % m;
      Ws[e] = W[i * ld + perm[r]];
    }
    __syncthreads();
    uint16_t* uo = p.u_out + (int64_t)s * p.out_stride;
    uint16_t* vo = p.v_out + (int64_t)s * p.out_stride;
    if (tall && D >= m) {  // W_m through the free Z region, and both products on the tensor cores
      for (int e = threadIdx.x; e < kp * m; e += THREADS) Z[e] = kAligned ? tf32_rn(Ws[e]) : Ws[e];
      __syncthreads();
      if constexpr (kAligned) {
        gemm_tall_tma<uint16_t, false, false>(T, m, kp, &p.maps[MAP_Y_MN], blockIdx.x, &p.maps[MAP_W_MN], blockIdx.x,
                                              uo, m, 1, ring, &tcs, tcur);  // U_m = Q W_m
        gemm_tall_tma<uint16_t, false, false>(D, m, kp, &p.maps[MAP_B_MN], blockIdx.x, &p.maps[MAP_W_MN], blockIdx.x,
                                              vo, m, 1, ring, &tcs, tcur);  // V_m = B^T W_m
      } else {
        gemm_tall<uint16_t, false, false, false, false>(T, m, kp, Y, T, Z, m, uo, m, 1, ring);  // U_m = Q W_m
        gemm_tall<uint16_t, false, false, false, false>(D, m, kp, B, D, Z, m, vo, m, 1, ring);  // V_m = B^T W_m
      }
    } else {
      gemm<uint16_t, false, false, false>(T, m, kp, Y, 1, T, Ws, m, 1, uo, m, 1, sA, sB);  // U_m = Q W_m
      gemm<uint16_t, false, false, false>(D, m, kp, B, 1, D, Ws, m, 1, vo, m, 1, sA, sB);  // V_m = B^T W_m
    }
  }
  if (kAligned && tall) tc_teardown(&tcs);
}

__host__ __device__ constexpr uint32_t factor_smem_bytes(int kp, int m) {
  return (uint32_t)sizeof(float) * (uint32_t)factor_smem_floats(kp, m);
}

}  // namespace factor
}  // namespace kamera
