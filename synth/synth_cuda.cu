// synth_cuda.cu -- device twin of synth/gen.py (seeded synthetic inputs).
//
// Input generation only: no arithmetic of the reuse operator lives here.  The
// values are bit-identical to gen.fill_rows (splitmix64 counter hash,
// Irwin-Hall sum of four 16-bit fields, one fp32 multiply, bf16 round to
// nearest even); a GPU test compares the two.  Used by the tests and the
// benchmark to fill multi-GB chunk stores on the device in milliseconds.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t hash64(uint64_t stream, uint64_t idx) {
  return mix64(stream + (idx + 1ull) * 0x9E3779B97F4A7C15ull);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  uint32_t u = __float_as_uint(x);
  u = u + 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

struct FillArgs {
  uint16_t* out;
  int64_t n_slabs, rows, row_len;
  int64_t out_slab_stride, out_row_stride;
  uint64_t stream, idx0, idx_slab_stride, idx_row_stride;
  float scale;
  uint64_t outlier_stream, okey0, okey_slab_stride;
  float outlier_scale;
  int32_t outlier_permille;
};

__global__ void fill_rows_kernel(FillArgs a) {
  const int64_t per_slab = a.rows * a.row_len;
  const int64_t total = a.n_slabs * per_slab;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t s = e / per_slab;
    const int64_t rem = e - s * per_slab;
    const int64_t r = rem / a.row_len;
    const int64_t j = rem - r * a.row_len;
    const uint64_t idx = a.idx0 + (uint64_t)s * a.idx_slab_stride + (uint64_t)r * a.idx_row_stride + (uint64_t)j;
    const uint64_t h = hash64(a.stream, idx);
    const uint32_t sum = (uint32_t)(h & 0xFFFFu) + (uint32_t)((h >> 16) & 0xFFFFu) + (uint32_t)((h >> 32) & 0xFFFFu) +
                         (uint32_t)(h >> 48);
    float scale = a.scale;
    if (a.outlier_permille > 0) {
      const uint64_t hk = hash64(a.outlier_stream, a.okey0 + (uint64_t)s * a.okey_slab_stride + (uint64_t)j);
      if ((int32_t)(hk % 1000ull) < a.outlier_permille) scale = a.outlier_scale;
    }
    const float x = (float)((int32_t)sum - 131070);
    a.out[s * a.out_slab_stride + r * a.out_row_stride + j] = f32_to_bf16_bits(__fmul_rn(x, scale));
  }
}

}  // namespace

extern "C" int synth_fill_rows(uint16_t* out, int64_t n_slabs, int64_t rows, int64_t row_len,
                               int64_t out_slab_stride, int64_t out_row_stride, uint64_t stream, uint64_t idx0,
                               uint64_t idx_slab_stride, uint64_t idx_row_stride, float scale,
                               uint64_t outlier_stream, uint64_t okey0, uint64_t okey_slab_stride,
                               float outlier_scale, int32_t outlier_permille, void* cuda_stream) {
  const int64_t total = n_slabs * rows * row_len;
  if (total <= 0) return 0;
  FillArgs a{out, n_slabs, rows, row_len, out_slab_stride, out_row_stride, stream, idx0, idx_slab_stride,
             idx_row_stride, scale, outlier_stream, okey0, okey_slab_stride, outlier_scale, outlier_permille};
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_rows_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>(a);
  return (int)cudaGetLastError();
}
