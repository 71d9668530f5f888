// Vocabulary-sharded argmax merge (page "radiance_drafthead.py": module docstring, where the head
// is x[M, 5120] @ W[5120, 124160] on each rank, and the launch-geometry notes that time one
// rank's vocab shard). With the head's vocab rows split across ranks at 64-row block boundaries, each
// rank runs the whole path on its shard; its blocks' candidates are exactly the unsharded head's
// blocks' candidates, so the only exchange is one per hidden row: the shard's best reranked
// (logit, vocab id). Each shard turns it into one 64-bit key whose signed integer order is the
// order (logit ascending, then id descending); the largest key over the shards -- a MAX
// all-reduce of int64 keys (NCCL, gloo), or a max over gathered keys -- names the global argmax
// with equal logits going to the lowest vocab id, the tie rule of the unsharded argmax.
//
// key = ((uint64 order_key(logit)) << 32 | (0xFFFFFFFF - global_id)) with the top bit flipped so
// that signed comparison matches unsigned. A row with no candidate at all gets INT64_MIN.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "dh_launch.h"

namespace dh {

namespace {

constexpr int64_t kNoKey = INT64_MIN;

__host__ __device__ inline uint32_t key_bits_of(float f) {
  uint32_t u;
#ifdef __CUDA_ARCH__
  u = __float_as_uint(f);
#else
  std::memcpy(&u, &f, sizeof u);
#endif
  if ((u & 0x7fffffffu) == 0u) u = 0u;  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__host__ __device__ inline float float_of_key_bits(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  float f;
#ifdef __CUDA_ARCH__
  f = __uint_as_float(u);
#else
  std::memcpy(&f, &u, sizeof f);
#endif
  return f;
}
// The shard key of (logit, global id); id in [0, 2^32 - 1).
__host__ __device__ inline int64_t make_key(float logit, int64_t id) {
  const uint64_t k = (static_cast<uint64_t>(key_bits_of(logit)) << 32) |
                     static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
  return static_cast<int64_t>(k ^ 0x8000000000000000ull);
}
__host__ __device__ inline void decode_key(int64_t key, int32_t* id, float* logit) {
  if (key == kNoKey) {
    *id = -1;
    *logit = -INFINITY;
    return;
  }
  const uint64_t k = static_cast<uint64_t>(key) ^ 0x8000000000000000ull;
  *id = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFu));
  *logit = float_of_key_bits(static_cast<uint32_t>(k >> 32));
}
// Best key of one hidden row's reranked list: slots with an id < 0 (empty) are skipped.
__host__ __device__ inline int64_t row_key(const int32_t* rr_id, const float* rr_logit, int R,
                                           int64_t id_offset) {
  int64_t best = kNoKey;
  for (int j = 0; j < R; ++j) {
    if (rr_id[j] < 0) continue;
    const int64_t k = make_key(rr_logit[j], rr_id[j] + id_offset);
    best = k > best ? k : best;
  }
  return best;
}

__global__ void shard_keys_kernel(const int32_t* rr_id, const float* rr_logit, int64_t M, int R,
                                  int64_t id_offset, int64_t* keys) {
  for (int64_t m = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; m < M;
       m += static_cast<int64_t>(gridDim.x) * blockDim.x)
    keys[m] = row_key(rr_id + m * R, rr_logit + m * R, R, id_offset);
}

__global__ void merge_keys_kernel(const int64_t* keys, int P, int64_t M, int32_t* argmax_id,
                                  float* logit) {
  for (int64_t m = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; m < M;
       m += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t best = kNoKey;
    for (int p = 0; p < P; ++p) {
      const int64_t k = keys[p * M + m];
      best = k > best ? k : best;
    }
    float v;
    int32_t id;
    decode_key(best, &id, &v);
    argmax_id[m] = id;
    if (logit) logit[m] = v;
  }
}

int grid_for(int64_t M) {
  const int64_t g = (M + 127) / 128;
  return static_cast<int>(g < 1024 ? g : 1024);
}

}  // namespace

cudaError_t launch_shard_keys(const int32_t* rr_id, const float* rr_logit, int64_t M, int R,
                              int64_t id_offset, int64_t* keys, cudaStream_t s) {
  shard_keys_kernel<<<grid_for(M), 128, 0, s>>>(rr_id, rr_logit, M, R, id_offset, keys);
  return cudaGetLastError();
}

cudaError_t launch_merge_keys(const int64_t* keys, int P, int64_t M, int32_t* argmax_id,
                              float* logit, cudaStream_t s) {
  merge_keys_kernel<<<grid_for(M), 128, 0, s>>>(keys, P, M, argmax_id, logit);
  return cudaGetLastError();
}

void shard_keys_host(const int32_t* rr_id, const float* rr_logit, int64_t M, int R,
                     int64_t id_offset, int64_t* keys) {
  for (int64_t m = 0; m < M; ++m) keys[m] = row_key(rr_id + m * R, rr_logit + m * R, R, id_offset);
}

void merge_keys_host(const int64_t* keys, int P, int64_t M, int32_t* argmax_id, float* logit) {
  for (int64_t m = 0; m < M; ++m) {
    int64_t best = kNoKey;
    for (int p = 0; p < P; ++p) best = keys[p * M + m] > best ? keys[p * M + m] : best;
    float v;
    decode_key(best, &argmax_id[m], &v);
    if (logit) logit[m] = v;
  }
}

}  // namespace dh
