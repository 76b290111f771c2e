// kamera_factor_general.cu -- the patch-formation kernel instance with run-time
// fallbacks for any shape, factor_kernel<false>, and its launch (see
// kamera_factor_launch.h).
#include "kamera_factor_launch.h"

namespace kamera {
namespace factor {

cudaError_t set_smem_limit_general(int bytes) {
  return cudaFuncSetAttribute(factor_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_general(const FParams& fp, int grid, uint32_t smem, cudaStream_t stream) {
  factor_kernel<false><<<grid, THREADS, smem, stream>>>(fp);
  return cudaGetLastError();
}

}  // namespace factor
}  // namespace kamera
