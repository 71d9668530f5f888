// Coarse-pass kernels for int2, G = 128 (one translation unit per variant: parallel builds).
#include "coarse_kernel.cuh"

namespace dh {

cudaError_t launch_coarse_i2g128(const CoarseArgs& a, int nsw, int grid, cudaStream_t s) {
  return launch_coarse_variant<2, 128>(a, nsw, grid, s);
}

}  // namespace dh
