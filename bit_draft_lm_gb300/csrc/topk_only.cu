// Logits for a top-K caller (page "radiance_drafthead.py", its top-K-only output of the head
// application): every entry of the row is -inf except the RERANK reranked ones, which
// carry their exact logit rounded to bf16, so a top-K request draws from the reranked pool only.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dh_device.cuh"
#include "dh_launch.h"

namespace dh {

constexpr int kTkThreads = 256;
constexpr int kTkChunk = 4096;  // row entries per CTA

// CTA (chunk, m): fills entries [chunk * kTkChunk, +kTkChunk) of row m with -inf, then writes
// the reranked entries that fall in that range (each entry has one writer: no race).
__global__ void __launch_bounds__(kTkThreads) topk_only_kernel(const int32_t* rr_id,
                                                               const float* rr_logit, int R,
                                                               int64_t N, uint16_t* y) {
  const int64_t m = blockIdx.y;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTkChunk;
  const int64_t n1 = n0 + kTkChunk < N ? n0 + kTkChunk : N;
  uint16_t* row = y + m * N;
  for (int64_t n = n0 + threadIdx.x; n < n1; n += kTkThreads) row[n] = 0xFF80u;  // bf16 -inf
  __syncthreads();
  for (int j = threadIdx.x; j < R; j += kTkThreads) {
    const int32_t id = rr_id[m * R + j];
    if (id >= n0 && id < n1)
      row[id] = __bfloat16_as_ushort(__float2bfloat16_rn(rr_logit[m * R + j]));
  }
}

cudaError_t launch_topk_only(const int32_t* rr_id, const float* rr_logit, int64_t M, int R,
                             int64_t N, void* y, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((N + kTkChunk - 1) / kTkChunk), static_cast<unsigned>(M));
  topk_only_kernel<<<grid, kTkThreads, 0, s>>>(rr_id, rr_logit, R, N, static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

}  // namespace dh
