// Coarse-pass kernels for int4, G = 128 (one translation unit per variant: parallel builds).
#include "coarse_kernel.cuh"

namespace dh {

cudaError_t launch_coarse_i4g128(const CoarseArgs& a, int nsw, int grid, cudaStream_t s) {
  return launch_coarse_variant<4, 128>(a, nsw, grid, s);
}

}  // namespace dh
