// C ABI of the draft head (include/drafthead.h): argument validation, launch, error reporting.
// No function here allocates device memory or synchronises, except dh_workspace_status.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>

#include "drafthead.h"

#include "dh_launch.h"

namespace {

constexpr size_t kWorkspaceHeader = 256;  // status word + reserved

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return DH_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DH_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceInfo {
  int sms = 0;
  int max_smem = 0;
};

// SM count and opt-in shared memory of the current device (looked up once per device).
cudaError_t device_info(DeviceInfo& out) {
  static DeviceInfo cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev].sms > 0) {
    out = cache[dev];
    return cudaSuccess;
  }
  DeviceInfo d;
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = d;
  out = d;
  return cudaSuccess;
}

int check_quant(const void* W, int64_t N, int64_t K, int G, const uint8_t* packed, const void* S,
                const void* ZS, int bits) {
  if (!W || !packed || !S || !ZS) return fail(DH_ERR_NULL, "quantize_pack: NULL pointer");
  if (G != 64 && G != 128) return fail(DH_ERR_PARAM, "quantize_pack: G=%d (64 or 128)", G);
  if (N < 1 || N > (int64_t)INT32_MAX || K < 1)
    return fail(DH_ERR_SHAPE, "quantize_pack: N=%lld K=%lld", (long long)N, (long long)K);
  const int64_t per = bits == 2 ? 4 : 2;
  if (K % (per * G))
    return fail(DH_ERR_SHAPE, "quantize_pack int%d: K=%lld must be a multiple of %lld", bits,
                (long long)K, (long long)(per * G));
  if (K > 32768) return fail(DH_ERR_SHAPE, "quantize_pack: K=%lld > 32768", (long long)K);
  if (!aligned(W, 16)) return fail(DH_ERR_ALIGN, "quantize_pack: W not 16-byte aligned");
  if (!aligned(packed, 4) || !aligned(S, 2) || !aligned(ZS, 2))
    return fail(DH_ERR_ALIGN, "quantize_pack: output misaligned (packed 4 B, S/ZS 2 B)");
  return DH_OK;
}

int quantize(int bits, const void* W, int64_t N, int64_t K, int G, uint8_t* packed, void* S,
             void* ZS, dh_stream_t s) {
  int rc = check_quant(W, N, K, G, packed, S, ZS, bits);
  if (rc != DH_OK) return rc;
  cudaError_t e = dh::launch_quantize_pack(bits, W, N, K, G, packed, S, ZS,
                                           reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "quantize_pack launch");
  return ok();
}

// The rerank needs the status word only; the coarse pass of more than kWideMinRows hidden rows
// also keeps its scratch after the header.
size_t rerank_workspace_bytes() { return kWorkspaceHeader; }
size_t coarse_workspace_bytes(int64_t M, int64_t K) {
  return kWorkspaceHeader + dh::coarse_wide_scratch_bytes(M, K);
}

int check_workspace(void* ws, size_t ws_bytes, size_t need, const char* who) {
  if (!ws) return fail(DH_ERR_WORKSPACE, "%s: workspace is NULL", who);
  if (!aligned(ws, 256)) return fail(DH_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", who);
  if (ws_bytes < need)
    return fail(DH_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu required", who, ws_bytes, need);
  return DH_OK;
}

}  // namespace

namespace dh {
// Records `msg` as the calling thread's dh_last_error() message and returns `code` (for entry
// points defined in other files of the library).
int record_error(int code, const char* msg) { return fail(code, "%s", msg); }
// Workspace bytes the rerank entry point requires (the status word's header).
size_t rerank_workspace_needed() { return rerank_workspace_bytes(); }
}  // namespace dh

extern "C" {

int dh_quantize_pack_int2(const void* W, int64_t N, int64_t K, int G, uint8_t* packed, void* S,
                          void* ZS, dh_stream_t s) {
  return quantize(2, W, N, K, G, packed, S, ZS, s);
}

int dh_quantize_pack_int4(const void* W, int64_t N, int64_t K, int G, uint8_t* packed, void* S,
                          void* ZS, dh_stream_t s) {
  return quantize(4, W, N, K, G, packed, S, ZS, s);
}

size_t dh_packed_bytes(int64_t N, int64_t K, int G, int bits) {
  if (N < 1 || K < 1 || (G != 64 && G != 128) || (bits != 2 && bits != 4)) return 0;
  const int64_t per = bits == 2 ? 4 : 2;
  if (K % (per * G)) return 0;
  return static_cast<size_t>(N) * static_cast<size_t>(K / per) +
         2 * static_cast<size_t>(N) * static_cast<size_t>(K / G) * 2;
}

size_t dh_workspace_bytes(int64_t M, int64_t N, int64_t K, int kcand, int rerank) {
  (void)N;
  (void)kcand;
  (void)rerank;
  if (M < 1 || K < 1) return 0;
  const size_t c = coarse_workspace_bytes(M, K), r = rerank_workspace_bytes();
  return c > r ? c : r;
}

int dh_draft_head_coarse_topk(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                              const void* S, const void* ZS, int64_t N, int G, int bits,
                              int kcand, float* cand_val, int32_t* cand_id, void* y_coarse,
                              void* workspace, size_t ws_bytes, dh_stream_t s) {
  const char* who = "draft_head_coarse_topk";
  if (!x || !packed || !S || !ZS || !cand_val || !cand_id)
    return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  if (bits != 2 && bits != 4) return fail(DH_ERR_PARAM, "%s: bits=%d (2 or 4)", who, bits);
  if (G != 64 && G != 128) return fail(DH_ERR_PARAM, "%s: G=%d (64 or 128)", who, G);
  if (kcand < 1 || kcand > DH_MAX_KCAND)
    return fail(DH_ERR_PARAM, "%s: kcand=%d (1..%d)", who, kcand, DH_MAX_KCAND);
  if (M < 1 || M > DH_MAX_TOKENS)
    return fail(DH_ERR_SHAPE, "%s: M=%lld (1..%d)", who, (long long)M, DH_MAX_TOKENS);
  if (N < 1 || N > (int64_t)INT32_MAX - DH_BLOCK_ROWS)
    return fail(DH_ERR_SHAPE, "%s: N=%lld", who, (long long)N);
  if (K < 8 * G || K % (8 * G) || K > 5120)
    return fail(DH_ERR_SHAPE, "%s: K=%lld must be a multiple of 8*G=%d and at most 5120", who,
                (long long)K, 8 * G);
  const int64_t nblk = (N + DH_BLOCK_ROWS - 1) / DH_BLOCK_ROWS;
  if (M * nblk * kcand > (int64_t)INT32_MAX)
    return fail(DH_ERR_SHAPE, "%s: M*nblk*kcand exceeds 2^31", who);
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(S, 16) || !aligned(ZS, 16))
    return fail(DH_ERR_ALIGN, "%s: x, packed, S and ZS must be 16-byte aligned", who);
  if (!aligned(cand_val, 4) || !aligned(cand_id, 4) || (y_coarse && !aligned(y_coarse, 2)))
    return fail(DH_ERR_ALIGN, "%s: output misaligned", who);
  int rc = check_workspace(workspace, ws_bytes, coarse_workspace_bytes(M, K), who);
  if (rc != DH_OK) return rc;
  DeviceInfo di;
  cudaError_t e = device_info(di);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  void* scratch = dh::coarse_wide_scratch_bytes(M, K)
                      ? static_cast<unsigned char*>(workspace) + kWorkspaceHeader
                      : nullptr;
  dh::CoarseCall cc{x,        M,       K,       packed,   S,
                    ZS,       N,       G,       bits,     kcand,
                    cand_val, cand_id, y_coarse, static_cast<uint32_t*>(workspace), scratch};
  e = dh::launch_coarse_topk(cc, di.sms, di.max_smem, reinterpret_cast<cudaStream_t>(s));
  if (e == cudaErrorInvalidValue)
    return fail(DH_ERR_SHAPE, "%s: shape does not fit the kernel's shared-memory plan", who);
  if (e != cudaSuccess) return cuda_fail(e, "coarse_topk launch");
  return ok();
}

int dh_draft_head_rerank_argmax(const void* x, int64_t M, int64_t K, const void* W, int64_t N,
                                const float* cand_val, const int32_t* cand_id, int64_t ncand,
                                int rerank, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                                void* y_coarse, void* workspace, size_t ws_bytes,
                                dh_stream_t s) {
  const char* who = "draft_head_rerank_argmax";
  if (!x || !W || !cand_val || !cand_id || !rr_id || !rr_logit || !argmax_id)
    return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  if (rerank < 1 || rerank > DH_MAX_RERANK)
    return fail(DH_ERR_PARAM, "%s: rerank=%d (1..%d)", who, rerank, DH_MAX_RERANK);
  if (M < 1 || M > DH_MAX_TOKENS)
    return fail(DH_ERR_SHAPE, "%s: M=%lld (1..%d)", who, (long long)M, DH_MAX_TOKENS);
  if (N < 1 || N > (int64_t)INT32_MAX || K < 8 || K % 8 || K > 32768)
    return fail(DH_ERR_SHAPE, "%s: N=%lld K=%lld (K a multiple of 8, at most 32768)", who,
                (long long)N, (long long)K);
  if (ncand < rerank || ncand > (int64_t)1 << 20)
    return fail(DH_ERR_SHAPE, "%s: ncand=%lld must be in [rerank, 2^20]", who, (long long)ncand);
  if (!aligned(x, 16) || !aligned(W, 16))
    return fail(DH_ERR_ALIGN, "%s: x and W must be 16-byte aligned", who);
  if (!aligned(cand_val, 4) || !aligned(cand_id, 4) || !aligned(rr_id, 4) ||
      !aligned(rr_logit, 4) || !aligned(argmax_id, 4) || (y_coarse && !aligned(y_coarse, 2)))
    return fail(DH_ERR_ALIGN, "%s: misaligned candidate or output array", who);
  int rc = check_workspace(workspace, ws_bytes, rerank_workspace_bytes(), who);
  if (rc != DH_OK) return rc;
  dh::RerankCall r{x, M, K, W, N, cand_val, cand_id, ncand, rerank, rr_id, rr_logit, argmax_id,
                   y_coarse, static_cast<uint32_t*>(workspace)};
  cudaError_t e = dh::launch_rerank_argmax(r, reinterpret_cast<cudaStream_t>(s));
  if (e == cudaErrorInvalidValue)
    return fail(DH_ERR_SHAPE, "%s: candidate count does not fit the kernel", who);
  if (e != cudaSuccess) return cuda_fail(e, "rerank_argmax launch");
  return ok();
}

int dh_workspace_status(const void* workspace, size_t ws_bytes, uint32_t* device_status,
                        dh_stream_t s) {
  if (!workspace || !device_status) return fail(DH_ERR_NULL, "workspace_status: NULL pointer");
  if (ws_bytes < sizeof(uint32_t)) return fail(DH_ERR_WORKSPACE, "workspace_status: too small");
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost,
                                  reinterpret_cast<cudaStream_t>(s));
  if (e == cudaSuccess) e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "workspace_status");
  *device_status = word;
  if (word) return fail(DH_ERR_DEVICE, "kernel status word 0x%x", word);
  return ok();
}

const char* dh_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
