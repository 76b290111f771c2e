// kamera_factor_aligned.cu -- the patch-formation kernel instance for aligned
// shapes, factor_kernel<true>, and its launch (see kamera_factor_launch.h).
#include "kamera_factor_launch.h"

namespace kamera {
namespace factor {

cudaError_t set_smem_limit_aligned(int bytes) {
  return cudaFuncSetAttribute(factor_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_aligned(const FParams& fp, int grid, uint32_t smem, cudaStream_t stream) {
  factor_kernel<true><<<grid, THREADS, smem, stream>>>(fp);
  return cudaGetLastError();
}

}  // namespace factor
}  // namespace kamera
