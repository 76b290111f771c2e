// kamera_factor_launch.h -- host entry points of the two patch-formation kernel
// instances.  Each instance is compiled in a translation unit of its own
// (kamera_factor_aligned.cu, kamera_factor_general.cu): they are by far the
// slowest code of the library to compile, and separate units build in
// parallel.  The host side (kamera_api.cu) calls only these functions; it never
// names the kernel template itself.
#pragma once
#include <cuda_runtime.h>

#include "kamera_factor.cuh"

namespace kamera {
namespace factor {

// factor_kernel<true>: T, D, k and the slab stride multiples of 4, Delta, Omega
// and the workspace 16-byte aligned (kamera_factor_aligned.cu).
cudaError_t set_smem_limit_aligned(int bytes);
cudaError_t launch_aligned(const FParams& fp, int grid, uint32_t smem, cudaStream_t stream);

// factor_kernel<false>: any shape, run-time fallbacks (kamera_factor_general.cu).
cudaError_t set_smem_limit_general(int bytes);
cudaError_t launch_general(const FParams& fp, int grid, uint32_t smem, cudaStream_t stream);

}  // namespace factor
}  // namespace kamera
