// Coarse-pass kernels for int4, G = 64 (one translation unit per variant: parallel builds).
#include "coarse_kernel.cuh"

namespace dh {

cudaError_t launch_coarse_i4g64(const CoarseArgs& a, int nsw, int grid, cudaStream_t s) {
  return launch_coarse_variant<4, 64>(a, nsw, grid, s);
}

}  // namespace dh
