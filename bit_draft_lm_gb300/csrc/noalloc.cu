// dh_draft_head_rerank_argmax_noalloc: the rerank + argmax call for callers that cannot allocate
// device memory (a plug-in that is handed only its input and output buffers, code that runs
// inside another framework's memory pool, or a caller whose allocator is unavailable at call
// time). The workspace the ordinary entry point takes from the caller lives here instead, in a
// fixed array among this library's device globals.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "drafthead.h"

#include "dh_launch.h"

namespace {

// The workspace of every call of dh_draft_head_rerank_argmax_noalloc on a device. Each device
// that loads the library holds DH_NOALLOC_SCRATCH_BYTES of it until the process exits.
// In host code this name denotes a host-side stand-in, not a device address: host code only
// ever passes the address that cudaGetSymbolAddress returns for it.
__device__ __align__(256) unsigned char g_noalloc_scratch[DH_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device, looked up once per device (with
// that device current).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dh::record_error(DH_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return dh::record_error(DH_ERR_CUDA, "draft_head_rerank_argmax_noalloc: device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "draft_head_rerank_argmax_noalloc: cudaGetSymbolAddress: %s",
               cudaGetErrorString(e));
      return dh::record_error(DH_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DH_OK;
}

}  // namespace

extern "C" int dh_draft_head_rerank_argmax_noalloc(const void* x, int64_t M, int64_t K,
                                                   const void* W, int64_t N, const float* cand_val,
                                                   const int32_t* cand_id, int64_t ncand,
                                                   int rerank, int32_t* rr_id, float* rr_logit,
                                                   int32_t* argmax_id, void* y_coarse,
                                                   dh_stream_t s) {
  const char* who = "draft_head_rerank_argmax_noalloc";
  // Every argument is checked first, with the checks of dh_draft_head_rerank_argmax (sizes out
  // of range: DH_ERR_SHAPE with a message), so that a refused call leaves nothing on the stream.
  int rc = dh::check_rerank_call(who, x, M, K, W, N, cand_val, cand_id, ncand, rerank, rr_id,
                                 rr_logit, argmax_id, y_coarse);
  if (rc != DH_OK) return rc;
  // The rerank's workspace is its status header, the same for every accepted size, so every
  // call the checks above accept fits in the array.
  const size_t need = dh::rerank_workspace_needed();
  if (need > DH_NOALLOC_SCRATCH_BYTES) {  // not reachable with the library's sizes
    char msg[200];
    snprintf(msg, sizeof msg, "%s: %zu bytes of workspace needed, more than the fixed %u-byte "
             "scratch", who, need, DH_NOALLOC_SCRATCH_BYTES);
    return dh::record_error(DH_ERR_SHAPE, msg);
  }
  void* ws = nullptr;
  rc = scratch_address(&ws);
  if (rc != DH_OK) return rc;
  // The array keeps the previous call's contents (status word included): start from zero.
  cudaError_t e = cudaMemsetAsync(ws, 0, need, reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "%s: clearing the scratch: %s", who, cudaGetErrorString(e));
    return dh::record_error(DH_ERR_CUDA, msg);
  }
  return dh_draft_head_rerank_argmax(x, M, K, W, N, cand_val, cand_id, ncand, rerank, rr_id,
                                     rr_logit, argmax_id, y_coarse, ws, DH_NOALLOC_SCRATCH_BYTES,
                                     s);
}
