// Host-side launch interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace dh {

struct CoarseCall {
  const void* x;
  int64_t M, K;
  const uint8_t* packed;
  const void* S;
  const void* ZS;
  int64_t N;
  int G, bits, kcand;
  float* cand_val;
  int32_t* cand_id;
  void* y;
  uint32_t* status;
  void* scratch;  // the coarse pass's part of the workspace (coarse_wide_scratch_bytes)
};

struct RerankCall {
  const void* x;
  int64_t M, K;
  const void* W;
  int64_t N;
  const float* cand_val;
  const int32_t* cand_id;
  int64_t ncand;
  int R;
  int32_t* rr_id;
  float* rr_logit;
  int32_t* argmax_id;
  void* y;
  uint32_t* status;
  const uint8_t* W8 = nullptr;      // e4m3 rows [N, K] instead of W (FP8 checkpoints) ...
  const float* wscale = nullptr;    // ... with their fp32 per-row scale [N]
  // device views of page-locked host arrays written with the same results (or nullptr)
  int32_t* h_rr_id = nullptr;
  float* h_rr_logit = nullptr;
  int32_t* h_argmax_id = nullptr;
};

// W bf16 [N, K], or (row_scale != nullptr) e4m3 [N, K] bytes whose values are multiplied by the
// fp32 per-row scale before quantising.
cudaError_t launch_quantize_pack(int bits, const void* W, int64_t N, int64_t K, int G,
                                 uint8_t* packed, void* S, void* ZS, cudaStream_t s,
                                 const float* row_scale = nullptr);
// cudaErrorInvalidValue: the shape does not fit the kernel's shared-memory plan.
cudaError_t launch_coarse_topk(const CoarseCall& cc, int num_sms, int max_smem, cudaStream_t s);
// The tensor-core (tcgen05) pass of int2 heads for more than kWideMinRows hidden rows, up to
// kWideMaxRows per pass (coarse_tc.cu). Its scratch (the hidden states laid out as the MMA
// operand, their group sums and scales) lives in the caller's workspace.
constexpr int kWideMinRows = 16;
constexpr int kWideMaxRows = 80;
size_t coarse_wide_scratch_bytes(int64_t M, int64_t K);
bool coarse_wide_supports(const CoarseCall& cc);
cudaError_t launch_coarse_wide(const CoarseCall& cc, void* scratch, int num_sms, int max_smem,
                               cudaStream_t s);
cudaError_t launch_rerank_argmax(const RerankCall& rc, cudaStream_t s);
// Copies `bytes` (a multiple of 16; both pointers 16-byte aligned) from src, the device view of
// page-locked host memory, to device memory; the next kernel in the stream may start its
// programmatic-dependent prologue meanwhile (host_io.cu).
cudaError_t launch_stage_in(const void* src, void* dst, size_t bytes, cudaStream_t s);
// y [M, N] bf16 = -inf except y[m, rr_id[m, j]] = bf16(rr_logit[m, j]) (topk_only.cu).
cudaError_t launch_topk_only(const int32_t* rr_id, const float* rr_logit, int64_t M, int R,
                             int64_t N, void* y, cudaStream_t s);
// Vocabulary-sharded argmax merge (shard_merge.cu): per-row int64 keys of a shard's reranked
// lists, and their merge over P shards ([P, M] keys) into global argmax ids and logits; device
// kernels and the same arithmetic on host arrays.
cudaError_t launch_shard_keys(const int32_t* rr_id, const float* rr_logit, int64_t M, int R,
                              int64_t id_offset, int64_t* keys, cudaStream_t s);
cudaError_t launch_merge_keys(const int64_t* keys, int P, int64_t M, int32_t* argmax_id,
                              float* logit, cudaStream_t s);
void shard_keys_host(const int32_t* rr_id, const float* rr_logit, int64_t M, int R,
                     int64_t id_offset, int64_t* keys);
void merge_keys_host(const int64_t* keys, int P, int64_t M, int32_t* argmax_id, float* logit);
// Sets the calling thread's dh_last_error() message; returns `code`.
int record_error(int code, const char* msg);
// Workspace bytes dh_draft_head_rerank_argmax requires (independent of the sizes).
size_t rerank_workspace_needed();
// dh_draft_head_rerank_argmax's argument checks (api.cu): DH_OK, or the failing check's status
// with its dh_last_error() message recorded.
int check_rerank_call(const char* who, const void* x, int64_t M, int64_t K, const void* W,
                      int64_t N, const float* cand_val, const int32_t* cand_id, int64_t ncand,
                      int rerank, int32_t* rr_id, float* rr_logit, int32_t* argmax_id,
                      void* y_coarse);

}  // namespace dh
