// C ABI of the draft head (include/drafthead.h): argument validation, launch, error reporting.
// No function here allocates device memory or synchronises, except dh_workspace_status.
#include <cuda_runtime.h>

#include <array>
#include <mutex>
#include <new>

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

// dh_draft_head_host: per device, a stream of the library's own for capturing (created on first
// use, kept until exit), and a small cache of captured graphs keyed by every argument.
struct HostGraphKey {
  std::array<uint64_t, 24> v;
};
struct HostGraph {
  HostGraphKey key{};
  cudaGraphExec_t exec = nullptr;
};
struct HostDevice {
  cudaStream_t stream = nullptr;  // where the graphs are captured
};
constexpr int kHostGraphs = 16;
std::mutex g_host_mu;
HostGraph g_host_graphs[kHostGraphs];
int g_host_next = 0;
HostDevice g_host_dev[64];

cudaError_t host_device(int dev, HostDevice** out) {
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  HostDevice& hd = g_host_dev[dev];
  if (hd.stream == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&hd.stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *out = &hd;
  return cudaSuccess;
}

}  // namespace

namespace dh {
// Records `msg` as the calling thread's dh_last_error() message and returns `code` (for entry
// points defined in other files of the library).
int record_error(int code, const char* msg) { return fail(code, "%s", msg); }
// Workspace bytes the rerank entry point requires (the status word's header).
size_t rerank_workspace_needed() { return rerank_workspace_bytes(); }
}  // namespace dh

static int check_rerank(const char* who, const void* x, int64_t M, int64_t K, const void* W,
                        const uint8_t* W8, const float* wscale, int64_t N, const float* cand_val,
                        const int32_t* cand_id, int64_t ncand, int rerank, int32_t* rr_id,
                        float* rr_logit, int32_t* argmax_id, void* y_coarse) {
  if (!x || (!W && !W8) || (W8 && !wscale) || !cand_val || !cand_id || !rr_id || !rr_logit || !argmax_id)
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
  if (!aligned(x, 16) || !aligned(W ? W : W8, 16) || (wscale && !aligned(wscale, 4)))
    return fail(DH_ERR_ALIGN, "%s: x and W must be 16-byte aligned", who);
  if (!aligned(cand_val, 4) || !aligned(cand_id, 4) || !aligned(rr_id, 4) ||
      !aligned(rr_logit, 4) || !aligned(argmax_id, 4) || (y_coarse && !aligned(y_coarse, 2)))
    return fail(DH_ERR_ALIGN, "%s: misaligned candidate or output array", who);
  return DH_OK;
}

namespace dh {
// The argument checks of dh_draft_head_rerank_argmax (bf16 rows), for the entry points defined in
// other files of the library; records the message and returns the status.
int check_rerank_call(const char* who, const void* x, int64_t M, int64_t K, const void* W,
                      int64_t N, const float* cand_val, const int32_t* cand_id, int64_t ncand,
                      int rerank, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                      void* y_coarse) {
  if (!W) return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  return check_rerank(who, x, M, K, W, nullptr, nullptr, N, cand_val, cand_id, ncand, rerank,
                      rr_id, rr_logit, argmax_id, y_coarse);
}
}  // namespace dh

static int rerank_impl(const char* who, const void* x, int64_t M, int64_t K, const void* W,
                       const uint8_t* W8, const float* wscale, int64_t N, const float* cand_val,
                       const int32_t* cand_id, int64_t ncand, int rerank, int32_t* rr_id,
                       float* rr_logit, int32_t* argmax_id, void* y_coarse, void* workspace,
                       size_t ws_bytes, dh_stream_t s) {
  int rc = check_rerank(who, x, M, K, W, W8, wscale, N, cand_val, cand_id, ncand, rerank, rr_id,
                        rr_logit, argmax_id, y_coarse);
  if (rc != DH_OK) return rc;
  rc = check_workspace(workspace, ws_bytes, rerank_workspace_bytes(), who);
  if (rc != DH_OK) return rc;
  dh::RerankCall r{x, M, K, W, N, cand_val, cand_id, ncand, rerank, rr_id, rr_logit, argmax_id,
                   y_coarse, static_cast<uint32_t*>(workspace), W8, wscale};
  cudaError_t e = dh::launch_rerank_argmax(r, reinterpret_cast<cudaStream_t>(s));
  if (e == cudaErrorInvalidValue)
    return fail(DH_ERR_SHAPE, "%s: candidate count does not fit the kernel", who);
  if (e != cudaSuccess) return cuda_fail(e, "rerank_argmax launch");
  return ok();
}

extern "C" {

int dh_quantize_pack_int2(const void* W, int64_t N, int64_t K, int G, uint8_t* packed, void* S,
                          void* ZS, dh_stream_t s) {
  return quantize(2, W, N, K, G, packed, S, ZS, s);
}

int dh_quantize_pack_int4(const void* W, int64_t N, int64_t K, int G, uint8_t* packed, void* S,
                          void* ZS, dh_stream_t s) {
  return quantize(4, W, N, K, G, packed, S, ZS, s);
}

int dh_quantize_pack_int2_fp8(const uint8_t* W8, const float* row_scale, int64_t N, int64_t K,
                              int G, uint8_t* packed, void* S, void* ZS, dh_stream_t s) {
  int rc = check_quant(W8, N, K, G, packed, S, ZS, 2);
  if (rc != DH_OK) return rc;
  if (!row_scale) return fail(DH_ERR_NULL, "quantize_pack_int2_fp8: row_scale is NULL");
  if (!aligned(row_scale, 4)) return fail(DH_ERR_ALIGN, "quantize_pack_int2_fp8: row_scale");
  cudaError_t e = dh::launch_quantize_pack(2, W8, N, K, G, packed, S, ZS,
                                           reinterpret_cast<cudaStream_t>(s), row_scale);
  if (e != cudaSuccess) return cuda_fail(e, "quantize_pack_int2_fp8 launch");
  return ok();
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

}  // extern "C"

static int check_coarse(const char* who, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const void* S, const void* ZS, int64_t N, int G,
                        int bits, int kcand, float* cand_val, int32_t* cand_id, void* y_coarse) {
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
  return DH_OK;
}

extern "C" {

int dh_draft_head_coarse_topk(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                              const void* S, const void* ZS, int64_t N, int G, int bits,
                              int kcand, float* cand_val, int32_t* cand_id, void* y_coarse,
                              void* workspace, size_t ws_bytes, dh_stream_t s) {
  const char* who = "draft_head_coarse_topk";
  int rc = check_coarse(who, x, M, K, packed, S, ZS, N, G, bits, kcand, cand_val, cand_id,
                        y_coarse);
  if (rc != DH_OK) return rc;
  rc = check_workspace(workspace, ws_bytes, coarse_workspace_bytes(M, K), who);
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
  if (!W) return fail(DH_ERR_NULL, "draft_head_rerank_argmax: NULL pointer");
  return rerank_impl("draft_head_rerank_argmax", x, M, K, W, nullptr, nullptr, N, cand_val,
                     cand_id, ncand, rerank, rr_id, rr_logit, argmax_id, y_coarse, workspace,
                     ws_bytes, s);
}

int dh_draft_head_rerank_argmax_fp8(const void* x, int64_t M, int64_t K, const uint8_t* W8,
                                    const float* row_scale, int64_t N, const float* cand_val,
                                    const int32_t* cand_id, int64_t ncand, int rerank,
                                    int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                                    void* y_coarse, void* workspace, size_t ws_bytes,
                                    dh_stream_t s) {
  if (!W8 || !row_scale) return fail(DH_ERR_NULL, "draft_head_rerank_argmax_fp8: NULL pointer");
  return rerank_impl("draft_head_rerank_argmax_fp8", x, M, K, nullptr, W8, row_scale, N,
                     cand_val, cand_id, ncand, rerank, rr_id, rr_logit, argmax_id, y_coarse,
                     workspace, ws_bytes, s);
}

}  // extern "C"

// dh_draft_head_argmax, optionally also writing the three results into page-locked host arrays
// through their device views (h_*: all three or none).
static int argmax_impl(const void* x, int64_t M, int64_t K, const uint8_t* packed, const void* S,
                       const void* ZS, const void* W, int64_t N, int G, int bits, int kcand,
                       int rerank, float* cand_val, int32_t* cand_id, int32_t* rr_id,
                       float* rr_logit, int32_t* argmax_id, void* y_coarse, void* workspace,
                       size_t ws_bytes, dh_stream_t s, int32_t* h_argmax_id = nullptr,
                       int32_t* h_rr_id = nullptr, float* h_rr_logit = nullptr) {
  const char* who = "draft_head_argmax";
  int rc = check_coarse(who, x, M, K, packed, S, ZS, N, G, bits, kcand, cand_val, cand_id,
                        y_coarse);
  if (rc != DH_OK) return rc;
  if (!W) return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  const int64_t ncand = ((N + DH_BLOCK_ROWS - 1) / DH_BLOCK_ROWS) * kcand;
  rc = check_rerank(who, x, M, K, W, nullptr, nullptr, N, cand_val, cand_id, ncand, rerank, rr_id,
                    rr_logit, argmax_id, y_coarse);
  if (rc != DH_OK) return rc;
  rc = check_workspace(workspace, ws_bytes, dh_workspace_bytes(M, N, K, kcand, rerank), who);
  if (rc != DH_OK) return rc;
  DeviceInfo di;
  cudaError_t e = device_info(di);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  void* scratch = dh::coarse_wide_scratch_bytes(M, K)
                      ? static_cast<unsigned char*>(workspace) + kWorkspaceHeader
                      : nullptr;
  uint32_t* status = static_cast<uint32_t*>(workspace);
  dh::CoarseCall cc{x,        M,       K,        packed, S,  ZS, N, G, bits, kcand,
                    cand_val, cand_id, y_coarse, status, scratch};
  e = dh::launch_coarse_topk(cc, di.sms, di.max_smem, cs);
  if (e == cudaErrorInvalidValue)
    return fail(DH_ERR_SHAPE, "%s: shape does not fit the kernel's shared-memory plan", who);
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_argmax coarse launch");
  // the rerank's cluster kernel starts as a programmatic dependent of the coarse pass: it stages
  // x while the coarse pass finishes and waits for the candidates
  dh::RerankCall r{x,       M,     K,      W,     N,        cand_val,  cand_id,
                   ncand,   rerank, rr_id, rr_logit, argmax_id, y_coarse, status};
  r.h_rr_id = h_rr_id;
  r.h_rr_logit = h_rr_logit;
  r.h_argmax_id = h_argmax_id;
  e = dh::launch_rerank_argmax(r, cs);
  if (e == cudaErrorInvalidValue)
    return fail(DH_ERR_SHAPE, "%s: candidate count does not fit the rerank kernel", who);
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_argmax rerank launch");
  return ok();
}

extern "C" {

int dh_draft_head_argmax(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                         const void* S, const void* ZS, const void* W, int64_t N, int G, int bits,
                         int kcand, int rerank, float* cand_val, int32_t* cand_id, int32_t* rr_id,
                         float* rr_logit, int32_t* argmax_id, void* y_coarse, void* workspace,
                         size_t ws_bytes, dh_stream_t s) {
  return argmax_impl(x, M, K, packed, S, ZS, W, N, G, bits, kcand, rerank, cand_val, cand_id,
                     rr_id, rr_logit, argmax_id, y_coarse, workspace, ws_bytes, s);
}

int dh_topk_only_logits(const int32_t* rr_id, const float* rr_logit, int64_t M, int rerank,
                        int64_t N, void* y, dh_stream_t s) {
  const char* who = "topk_only_logits";
  if (!rr_id || !rr_logit || !y) return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  if (M < 1 || M > DH_MAX_TOKENS || N < 1 || N > (int64_t)INT32_MAX || rerank < 1 ||
      rerank > DH_MAX_RERANK)
    return fail(DH_ERR_SHAPE, "%s: M=%lld N=%lld rerank=%d", who, (long long)M, (long long)N,
                rerank);
  if (!aligned(rr_id, 4) || !aligned(rr_logit, 4) || !aligned(y, 2))
    return fail(DH_ERR_ALIGN, "%s: misaligned array", who);
  cudaError_t e = dh::launch_topk_only(rr_id, rr_logit, M, rerank, N, y,
                                       reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "topk_only_logits launch");
  return ok();
}

}  // extern "C"

// ---- vocabulary-sharded argmax merge -------------------------------------------------------------
static int check_shard_keys(const char* who, const int32_t* rr_id, const float* rr_logit,
                            int64_t M, int rerank, int64_t id_offset, const int64_t* keys) {
  if (!rr_id || !rr_logit || !keys) return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  if (M < 1 || M > DH_MAX_TOKENS || rerank < 1 || rerank > DH_MAX_RERANK)
    return fail(DH_ERR_SHAPE, "%s: M=%lld rerank=%d", who, (long long)M, rerank);
  if (id_offset < 0 || id_offset > (int64_t)INT32_MAX)
    return fail(DH_ERR_SHAPE, "%s: id_offset=%lld (0..2^31-1)", who, (long long)id_offset);
  if (!aligned(rr_id, 4) || !aligned(rr_logit, 4) || !aligned(keys, 8))
    return fail(DH_ERR_ALIGN, "%s: misaligned array", who);
  return DH_OK;
}

static int check_merge(const char* who, const int64_t* keys, int P, int64_t M,
                       const int32_t* argmax_id, const float* logit) {
  if (!keys || !argmax_id) return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  if (P < 1 || P > 65536 || M < 1 || M > DH_MAX_TOKENS)
    return fail(DH_ERR_SHAPE, "%s: P=%d M=%lld", who, P, (long long)M);
  if (!aligned(keys, 8) || !aligned(argmax_id, 4) || (logit && !aligned(logit, 4)))
    return fail(DH_ERR_ALIGN, "%s: misaligned array", who);
  return DH_OK;
}

extern "C" {

int dh_argmax_shard_keys(const int32_t* rr_id, const float* rr_logit, int64_t M, int rerank,
                         int64_t id_offset, int64_t* keys, dh_stream_t s) {
  const char* who = "argmax_shard_keys";
  int rc = check_shard_keys(who, rr_id, rr_logit, M, rerank, id_offset, keys);
  if (rc != DH_OK) return rc;
  cudaError_t e = dh::launch_shard_keys(rr_id, rr_logit, M, rerank, id_offset, keys,
                                        reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "argmax_shard_keys launch");
  return ok();
}

int dh_argmax_merge(const int64_t* keys, int P, int64_t M, int32_t* argmax_id, float* logit,
                    dh_stream_t s) {
  const char* who = "argmax_merge";
  int rc = check_merge(who, keys, P, M, argmax_id, logit);
  if (rc != DH_OK) return rc;
  cudaError_t e =
      dh::launch_merge_keys(keys, P, M, argmax_id, logit, reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "argmax_merge launch");
  return ok();
}

int dh_argmax_shard_keys_host(const int32_t* rr_id, const float* rr_logit, int64_t M, int rerank,
                              int64_t id_offset, int64_t* keys) {
  int rc = check_shard_keys("argmax_shard_keys_host", rr_id, rr_logit, M, rerank, id_offset, keys);
  if (rc != DH_OK) return rc;
  dh::shard_keys_host(rr_id, rr_logit, M, rerank, id_offset, keys);
  return ok();
}

int dh_argmax_merge_host(const int64_t* keys, int P, int64_t M, int32_t* argmax_id,
                         float* logit) {
  int rc = check_merge("argmax_merge_host", keys, P, M, argmax_id, logit);
  if (rc != DH_OK) return rc;
  dh::merge_keys_host(keys, P, M, argmax_id, logit);
  return ok();
}

}  // extern "C"

// Checks of the host-memory call's own arguments (the device calls it makes check the rest).
static int check_host(const char* who, const void* x_host, int64_t M, int64_t K, void* x_dev,
                      int rerank, int32_t* argmax_host, int32_t* rr_id_host,
                      float* rr_logit_host) {
  if (!x_host || !x_dev || !argmax_host || !rr_id_host || !rr_logit_host)
    return fail(DH_ERR_NULL, "%s: NULL pointer", who);
  if (M < 1 || M > DH_MAX_TOKENS || K < 1 || rerank < 1 || rerank > DH_MAX_RERANK)
    return fail(DH_ERR_SHAPE, "%s: M=%lld K=%lld rerank=%d", who, (long long)M, (long long)K,
                rerank);
  if (!aligned(x_dev, 16)) return fail(DH_ERR_ALIGN, "%s: x_dev must be 16-byte aligned", who);
  return DH_OK;
}

static int check_not_capturing(const char* who, cudaStream_t us) {
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(us, &cap_status);
  if (e != cudaSuccess) return cuda_fail(e, "stream query");
  if (cap_status != cudaStreamCaptureStatusNone)
    return fail(DH_ERR_PARAM, "%s: the stream is being captured (this call synchronises)", who);
  return DH_OK;
}

// The host-memory call captured into an executable graph on device dev's capture stream (a
// capture cannot run on the legacy default stream). Caller holds g_host_mu.
static int capture_host_call(int dev, const void* x_host, int64_t M, int64_t K, void* x_dev,
                             const uint8_t* packed, const void* S, const void* ZS, const void* W,
                             int64_t N, int G, int bits, int kcand, int rerank, float* cand_val,
                             int32_t* cand_id, int32_t* rr_id, float* rr_logit,
                             int32_t* argmax_id, int32_t* argmax_host, int32_t* rr_id_host,
                             float* rr_logit_host, void* workspace, size_t ws_bytes,
                             cudaGraphExec_t* out) {
  HostDevice* hd = nullptr;
  cudaError_t e = host_device(dev, &hd);
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_host: stream creation");
  const cudaStream_t cs = hd->stream;
  const size_t xb = static_cast<size_t>(M) * static_cast<size_t>(K) * 2;
  const size_t rb = static_cast<size_t>(M) * static_cast<size_t>(rerank) * 4;
  // Page-locked host arrays mapped into the device's address space: x is staged by a copy
  // kernel (the coarse pass starts during it, as its programmatic dependent) and the rerank
  // writes the results into the host arrays itself, so the graph holds kernels only.
  // Otherwise: copy-engine transfers in and out.
  void* xv = nullptr;
  void* av = nullptr;
  void* iv = nullptr;
  void* lv = nullptr;
  const bool mapped =
      cudaHostGetDevicePointer(&xv, const_cast<void*>(x_host), 0) == cudaSuccess &&
      cudaHostGetDevicePointer(&av, argmax_host, 0) == cudaSuccess &&
      cudaHostGetDevicePointer(&iv, rr_id_host, 0) == cudaSuccess &&
      cudaHostGetDevicePointer(&lv, rr_logit_host, 0) == cudaSuccess && aligned(xv, 16) &&
      xb % 16 == 0;
  if (!mapped) (void)cudaGetLastError();  // a failed lookup leaves no error behind
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_host: begin capture");
  int rc = DH_OK;
  const dh_stream_t ds = reinterpret_cast<dh_stream_t>(cs);
  if (mapped) {
    e = dh::launch_stage_in(xv, x_dev, xb, cs);
    if (e == cudaSuccess)
      rc = argmax_impl(x_dev, M, K, packed, S, ZS, W, N, G, bits, kcand, rerank, cand_val,
                       cand_id, rr_id, rr_logit, argmax_id, nullptr, workspace, ws_bytes, ds,
                       static_cast<int32_t*>(av), static_cast<int32_t*>(iv),
                       static_cast<float*>(lv));
  } else {
    e = cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
      rc = argmax_impl(x_dev, M, K, packed, S, ZS, W, N, G, bits, kcand, rerank, cand_val,
                       cand_id, rr_id, rr_logit, argmax_id, nullptr, workspace, ws_bytes, ds);
    if (e == cudaSuccess && rc == DH_OK) {
      // one copy when the three results lie back to back on both sides (argmax, rr_id,
      // rr_logit), else three
      const size_t ab = static_cast<size_t>(M) * 4;
      auto* dv = reinterpret_cast<const unsigned char*>(argmax_id);
      auto* hv = reinterpret_cast<unsigned char*>(argmax_host);
      const bool joint = reinterpret_cast<const unsigned char*>(rr_id) == dv + ab &&
                         reinterpret_cast<const unsigned char*>(rr_logit) == dv + ab + rb &&
                         reinterpret_cast<unsigned char*>(rr_id_host) == hv + ab &&
                         reinterpret_cast<unsigned char*>(rr_logit_host) == hv + ab + rb;
      if (joint) {
        e = cudaMemcpyAsync(hv, dv, ab + 2 * rb, cudaMemcpyDeviceToHost, cs);
      } else {
        e = cudaMemcpyAsync(argmax_host, argmax_id, ab, cudaMemcpyDeviceToHost, cs);
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(rr_id_host, rr_id, rb, cudaMemcpyDeviceToHost, cs);
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(rr_logit_host, rr_logit, rb, cudaMemcpyDeviceToHost, cs);
      }
    }
  }
  cudaGraph_t graph = nullptr;
  const cudaError_t ee = cudaStreamEndCapture(cs, &graph);
  if (rc != DH_OK || e != cudaSuccess || ee != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    if (rc != DH_OK) return rc;  // the failing call recorded its message
    return cuda_fail(e != cudaSuccess ? e : ee, "draft_head_host: capture");
  }
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_host: instantiate");
  *out = exec;
  return DH_OK;
}

// Replays an executable graph of the host-memory call on s and waits for it.
static int run_host_graph(cudaGraphExec_t exec, cudaStream_t us) {
  cudaError_t e = cudaGraphLaunch(exec, us);  // stream-ordered after the caller's earlier work
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_host: launch");
  e = cudaStreamSynchronize(us);
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_host: synchronise");
  return ok();
}

struct dh_host_plan_s {
  cudaGraphExec_t exec;
};

extern "C" {

int dh_draft_head_host(const void* x_host, int64_t M, int64_t K, void* x_dev,
                       const uint8_t* packed, const void* S, const void* ZS, const void* W,
                       int64_t N, int G, int bits, int kcand, int rerank, float* cand_val,
                       int32_t* cand_id, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                       int32_t* argmax_host, int32_t* rr_id_host, float* rr_logit_host,
                       void* workspace, size_t ws_bytes, dh_stream_t s) {
  const char* who = "draft_head_host";
  int rc = check_host(who, x_host, M, K, x_dev, rerank, argmax_host, rr_id_host, rr_logit_host);
  if (rc != DH_OK) return rc;
  cudaStream_t us = reinterpret_cast<cudaStream_t>(s);
  rc = check_not_capturing(who, us);
  if (rc != DH_OK) return rc;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "draft_head_host: device query");

  // The whole sequence once per distinct argument set and device, then replayed on s itself.
  HostGraphKey key{};
  const uint64_t vals[] = {reinterpret_cast<uint64_t>(x_host), static_cast<uint64_t>(M),
                           static_cast<uint64_t>(K), reinterpret_cast<uint64_t>(x_dev),
                           reinterpret_cast<uint64_t>(packed), reinterpret_cast<uint64_t>(S),
                           reinterpret_cast<uint64_t>(ZS), reinterpret_cast<uint64_t>(W),
                           static_cast<uint64_t>(N), static_cast<uint64_t>(G),
                           static_cast<uint64_t>(bits), static_cast<uint64_t>(kcand),
                           static_cast<uint64_t>(rerank), reinterpret_cast<uint64_t>(cand_val),
                           reinterpret_cast<uint64_t>(cand_id), reinterpret_cast<uint64_t>(rr_id),
                           reinterpret_cast<uint64_t>(rr_logit),
                           reinterpret_cast<uint64_t>(argmax_id),
                           reinterpret_cast<uint64_t>(argmax_host),
                           reinterpret_cast<uint64_t>(rr_id_host),
                           reinterpret_cast<uint64_t>(rr_logit_host),
                           reinterpret_cast<uint64_t>(workspace), static_cast<uint64_t>(ws_bytes),
                           static_cast<uint64_t>(dev)};
  static_assert(sizeof(vals) == sizeof(key.v), "key size");
  for (size_t i = 0; i < sizeof(vals) / sizeof(vals[0]); ++i) key.v[i] = vals[i];

  std::lock_guard<std::mutex> lock(g_host_mu);
  cudaGraphExec_t exec = nullptr;
  for (auto& c : g_host_graphs)
    if (c.exec && c.key.v == key.v) exec = c.exec;
  if (exec == nullptr) {
    rc = capture_host_call(dev, x_host, M, K, x_dev, packed, S, ZS, W, N, G, bits, kcand, rerank,
                           cand_val, cand_id, rr_id, rr_logit, argmax_id, argmax_host,
                           rr_id_host, rr_logit_host, workspace, ws_bytes, &exec);
    if (rc != DH_OK) return rc;
    HostGraph& slot = g_host_graphs[g_host_next];
    g_host_next = (g_host_next + 1) % kHostGraphs;
    if (slot.exec) cudaGraphExecDestroy(slot.exec);  // the oldest argument set
    slot.key = key;
    slot.exec = exec;
  }
  return run_host_graph(exec, us);
}

int dh_host_plan_create(const void* x_host, int64_t M, int64_t K, void* x_dev,
                        const uint8_t* packed, const void* S, const void* ZS, const void* W,
                        int64_t N, int G, int bits, int kcand, int rerank, float* cand_val,
                        int32_t* cand_id, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                        int32_t* argmax_host, int32_t* rr_id_host, float* rr_logit_host,
                        void* workspace, size_t ws_bytes, dh_host_plan* plan) {
  const char* who = "host_plan_create";
  if (!plan) return fail(DH_ERR_NULL, "%s: NULL plan pointer", who);
  *plan = nullptr;
  int rc = check_host(who, x_host, M, K, x_dev, rerank, argmax_host, rr_id_host, rr_logit_host);
  if (rc != DH_OK) return rc;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "host_plan_create: device query");
  dh_host_plan p = new (std::nothrow) dh_host_plan_s{nullptr};
  if (!p) return fail(DH_ERR_PARAM, "%s: out of host memory", who);
  {
    std::lock_guard<std::mutex> lock(g_host_mu);
    rc = capture_host_call(dev, x_host, M, K, x_dev, packed, S, ZS, W, N, G, bits, kcand, rerank,
                           cand_val, cand_id, rr_id, rr_logit, argmax_id, argmax_host,
                           rr_id_host, rr_logit_host, workspace, ws_bytes, &p->exec);
  }
  if (rc != DH_OK) {
    delete p;
    return rc;
  }
  *plan = p;
  return ok();
}

int dh_host_plan_run(dh_host_plan plan, dh_stream_t s) {
  if (!plan) return fail(DH_ERR_NULL, "host_plan_run: NULL plan");
  cudaStream_t us = reinterpret_cast<cudaStream_t>(s);
  const int rc = check_not_capturing("host_plan_run", us);
  if (rc != DH_OK) return rc;
  return run_host_graph(plan->exec, us);
}

void dh_host_plan_destroy(dh_host_plan plan) {
  if (!plan) return;
  cudaGraphExecDestroy(plan->exec);
  delete plan;
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
