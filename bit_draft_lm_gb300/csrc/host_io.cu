// Staging of the hidden states from page-locked host memory for the host-memory entry point:
// a small copy kernel instead of a copy-engine transfer, so that the coarse pass, launched as
// its programmatic dependent, prefetches its weights while x crosses the host link.
#include <cuda_runtime.h>

#include <cstdint>

#include "dh_device.cuh"
#include "dh_launch.h"

namespace dh {

__global__ void __launch_bounds__(256) stage_in_kernel(const uint4* __restrict__ src,
                                                       uint4* __restrict__ dst, int n16) {
  if (threadIdx.x == 0) grid_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += blockDim.x * gridDim.x)
    dst[i] = src[i];
}

cudaError_t launch_stage_in(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  if (bytes % 16 || reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16 ||
      bytes / 16 > static_cast<size_t>(INT32_MAX))
    return cudaErrorInvalidValue;
  const int n16 = static_cast<int>(bytes / 16);
  if (n16 == 0) return cudaSuccess;
  int blocks = (n16 + 255) / 256;
  blocks = blocks > 64 ? 64 : blocks;
  stage_in_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                         n16);
  return cudaGetLastError();
}

}  // namespace dh
