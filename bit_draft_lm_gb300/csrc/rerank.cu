// Global top-RERANK over the block candidates, exact rerank and argmax (page
// "radiance_drafthead.py": the head application's RERANK best candidates, the exact rerank with
// bf16 rows, and the argmax its caller takes), for sm_103a.
//
// One CTA (1024 threads) per hidden row m:
//  1. the row's candidates are held in registers (LPT per thread) as order-preserving keys;
//  2. selection, exact and deterministic (order: value descending, then lowest id, then lowest
//     slot index, i.e. the sort that defines the operation): a threshold T that provably lies
//     at or below the R-th largest value filters the candidates, the survivors are compacted to
//     shared memory and one warp sorts (<= 32) or selects (<= 256) them; with more survivors
//     (heavy ties) or R > 32, R rounds each retire the CTA-wide first remaining candidate;
//  3. rerank: 32/R warps per selected row over slices of K, 16-byte loads of the bf16 weight
//     row against the hidden row staged in shared memory, fp32 accumulation, xor-shuffle tree,
//     slice sums added in a fixed order;
//  4. argmax over the rescored values (ties to the lowest vocab id) and the optional scatter of
//     bf16(logit) into the coarse logits.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "dh_device.cuh"
#include "dh_launch.h"

namespace dh {

namespace cg = cooperative_groups;

constexpr int kRerankThreads = 1024;
constexpr int kRerankWarps = kRerankThreads / 32;

struct RerankArgs {
  const uint16_t* x;  // bf16 [M, K]
  int K, N;
  const uint16_t* W;  // bf16 [N, K] (bf16 rows)
  const uint8_t* W8;  // e4m3 [N, K] (FP8 rows) ...
  const float* wscale;  // ... and their fp32 per-row scale [N]
  const float* cand_val;  // [M, ncand]
  const int32_t* cand_id;
  int ncand, R;
  int32_t* rr_id;      // [M, R]
  float* rr_logit;     // [M, R]
  int32_t* argmax_id;  // [M]
  uint16_t* y;         // bf16 [M, N] or nullptr
  uint32_t* status;
  // device views of page-locked host arrays that receive the same three results, or nullptr
  int32_t* h_rr_id;
  float* h_rr_logit;
  int32_t* h_argmax_id;
};

// Selection order: key descending, then id ascending (as unsigned with the sign bit flipped),
// then slot index ascending.
struct Sel {
  uint32_t key, uid, idx;
};

__device__ __forceinline__ bool sel_before(const Sel& a, const Sel& b) {
  if (a.key != b.key) return a.key > b.key;
  if (a.uid != b.uid) return a.uid < b.uid;
  return a.idx < b.idx;
}

// Warp-wide best of one Sel per lane (all lanes get the result).
__device__ __forceinline__ Sel warp_best(const Sel& s) {
  Sel r;
  r.key = __reduce_max_sync(0xffffffffu, s.key);
  r.uid = __reduce_min_sync(0xffffffffu, s.key == r.key ? s.uid : 0xffffffffu);
  r.idx = __reduce_min_sync(0xffffffffu, (s.key == r.key && s.uid == r.uid) ? s.idx : 0xffffffffu);
  return r;
}

// Bitonic sort of one Sel per lane across the warp: lane 0 ends with the first in selection
// order. Empty lanes carry key 0 and sort last.
__device__ __forceinline__ Sel warp_sort(Sel v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      Sel o;
      o.key = __shfl_xor_sync(0xffffffffu, v.key, j);
      o.uid = __shfl_xor_sync(0xffffffffu, v.uid, j);
      o.idx = __shfl_xor_sync(0xffffffffu, v.idx, j);
      const bool keep_first = ((lane & j) == 0) == ((lane & k) == 0);
      const bool o_first = sel_before(o, v);
      if (keep_first == o_first) v = o;
    }
  }
  return v;
}

constexpr int kSurvivorCap = 256;  // candidates the one-warp exact selection takes after the filter
constexpr int kRerankUnroll = 8;   // weight-row loads each lane keeps in flight

// 8 weights of a row, k = 8 k8 .. 8 k8 + 7: 16 bytes of bf16 or 8 bytes of e4m3.
template <bool FP8>
struct Row8 {
  using Raw = typename std::conditional<FP8, uint2, uint4>::type;
};
__device__ __forceinline__ uint2 ldg_nc_v2(const uint2* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
// Weight pair q (k = 8 k8 + 2q, + 1) of 8 loaded weights, as fp32 (exact).
__device__ __forceinline__ void w_pair(const uint4& w, int q, float& lo, float& hi) {
  const uint32_t v = q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w;
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xffff0000u);
}
// e4m3 bytes: the page's exact bit decode of its FP8 rerank, no hardware conversion.
__device__ __forceinline__ void w_pair(const uint2& w, int q, float& lo, float& hi) {
  const uint32_t v = q < 2 ? w.x : w.y;
  const int sh = 16 * (q & 1);
  lo = e4m3_bits_to_f32((v >> sh) & 0xffu);
  hi = e4m3_bits_to_f32((v >> (sh + 8)) & 0xffu);
}
template <bool FP8>
__device__ __forceinline__ typename Row8<FP8>::Raw load_w8(const RerankArgs& a, int n, int k8);

// Loads through the read-only (non-coherent) path: W is never written by the library.
__device__ __forceinline__ uint4 ldg_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <>
__device__ __forceinline__ uint4 load_w8<false>(const RerankArgs& a, int n, int k8) {
  return ldg_nc_v4(reinterpret_cast<const uint4*>(a.W + static_cast<int64_t>(n) * a.K) + k8);
}
template <>
__device__ __forceinline__ uint2 load_w8<true>(const RerankArgs& a, int n, int k8) {
  return ldg_nc_v2(reinterpret_cast<const uint2*>(a.W8 + static_cast<int64_t>(n) * a.K) + k8);
}
// The factor the row's dot is multiplied by: 1 for bf16 rows, the per-row scale for e4m3 rows.
template <bool FP8>
__device__ __forceinline__ float row_scale(const RerankArgs& a, int n) {
  return FP8 ? a.wscale[n] : 1.0f;
}

template <int LPT, bool FP8>
__global__ void __launch_bounds__(kRerankThreads, 1) rerank_argmax_kernel(const RerankArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);                      // [K]
  Sel* wbest = reinterpret_cast<Sel*>(sm + 2 * a.K);                    // [32]
  Sel* chosen = wbest + kRerankWarps;                                   // [1]
  int32_t* sel_id = reinterpret_cast<int32_t*>(chosen + 1);             // [R]
  float* sel_logit = reinterpret_cast<float*>(sel_id + a.R);           // [R]
  float* part_logit = sel_logit + a.R;                                  // [R * wpr]
  Sel* surv = reinterpret_cast<Sel*>(part_logit + a.R * kRerankWarps);  // [kSurvivorCap]
  uint32_t* wtmp = reinterpret_cast<uint32_t*>(surv + kSurvivorCap);    // [32 + 2]
  uint32_t* retired = wtmp + kRerankWarps + 2;                          // [ncand/32] (LPT == 0)

  const int m = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint16_t* xrow = a.x + static_cast<int64_t>(m) * a.K;
  // the next kernel in the stream (the next call's coarse pass) may start its weight prefetch
  // on the SMs this small grid leaves idle; it waits for this grid before reading anything else
  if (tid == 0) grid_launch_dependents();

  const float* cv = a.cand_val + static_cast<int64_t>(m) * a.ncand;
  const int32_t* ci = a.cand_id + static_cast<int64_t>(m) * a.ncand;
  // LPT > 0: this thread's candidates live in registers; LPT == 0: candidates are re-read from
  // global memory every round and a shared bitmap marks the retired slots.
  // Only the keys stay in registers; ids are re-read (L1/L2) where a tie-break or a result
  // needs them.
  constexpr int kRegs = LPT > 0 ? LPT : 1;
  uint32_t key[kRegs];
  auto uid_at = [&](int i) { return static_cast<uint32_t>(ci[i]) ^ 0x80000000u; };
  if (LPT == 0)
    for (int i = tid; i < (a.ncand + 31) / 32; i += kRerankThreads) retired[i] = 0u;
#pragma unroll
  for (int j = 0; j < LPT; ++j) {
    const int i = tid + j * kRerankThreads;
    key[j] = i < a.ncand ? order_key(cv[i]) : 0u;
  }

  // the hidden row, staged for the rerank dots (its loads overlap those of the keys)
  for (int i = tid; i < a.K / 8; i += kRerankThreads)
    reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(xrow)[i];

  // Fast exact path. T = the R-th largest of the 32 warp maxima is at most the R-th largest
  // candidate (those R maxima are R distinct candidates >= T), so every member of the top R has
  // key >= T. Items >= T are compacted into shared memory and one warp selects among them.
  bool selected = false;
  if (LPT > 0 && a.R <= 32) {
    uint32_t tmax = 0u;
#pragma unroll
    for (int j = 0; j < kRegs; ++j) tmax = max(tmax, key[j]);
    tmax = __reduce_max_sync(0xffffffffu, tmax);
    if (lane == 0) wtmp[warp] = tmax;
    __syncthreads();
    if (warp == 0) {
      const Sel w = warp_sort(Sel{wtmp[lane], 0u, static_cast<uint32_t>(lane)});
      const uint32_t T = __shfl_sync(0xffffffffu, w.key, a.R - 1);
      if (lane == 0) wtmp[kRerankWarps] = T;
    }
    __syncthreads();
    const uint32_t T = wtmp[kRerankWarps];
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kRegs; ++j) cnt += (key[j] != 0u && key[j] >= T) ? 1 : 0;
    int incl = cnt;  // warp inclusive scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    __syncthreads();  // every thread has read T before wtmp is reused
    if (lane == 31) wtmp[warp] = static_cast<uint32_t>(incl);
    __syncthreads();
    if (warp == 0) {
      int wsum = static_cast<int>(wtmp[lane]);
      int wincl = wsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += v;
      }
      __syncwarp();
      wtmp[lane] = static_cast<uint32_t>(wincl - wsum);  // exclusive warp base
      if (lane == 31) wtmp[kRerankWarps + 1] = static_cast<uint32_t>(wincl);
    }
    __syncthreads();
    const int total = static_cast<int>(wtmp[kRerankWarps + 1]);
    if (total <= kSurvivorCap) {
      int pos = static_cast<int>(wtmp[warp]) + incl - cnt;
#pragma unroll
      for (int j = 0; j < kRegs; ++j)
        if (key[j] != 0u && key[j] >= T) {
          const int i = tid + j * kRerankThreads;
          surv[pos++] = Sel{key[j], uid_at(i), static_cast<uint32_t>(i)};
        }
    }
    __syncthreads();
    if (total <= kSurvivorCap) {
      selected = true;
      if (warp == 0) {
        if (total <= 32) {
          Sel v = lane < total ? surv[lane] : Sel{0u, 0xffffffffu, 0xffffffffu};
          v = warp_sort(v);
          if (lane < a.R) sel_id[lane] = static_cast<int32_t>(v.uid ^ 0x80000000u);
        } else {
          for (int r = 0; r < a.R; ++r) {
            Sel best{0u, 0xffffffffu, 0xffffffffu};
            for (int q = lane; q < total; q += 32) {
              const Sel v = surv[q];
              if (v.key != 0u && (best.key == 0u || sel_before(v, best))) best = v;
            }
            const Sel wb = warp_best(best);
            for (int q = lane; q < total; q += 32)
              if (surv[q].key != 0u && surv[q].idx == wb.idx) surv[q].key = 0u;
            __syncwarp();
            if (lane == 0) sel_id[r] = static_cast<int32_t>(wb.uid ^ 0x80000000u);
          }
        }
      }
    }
    __syncthreads();
  }

  for (int r = 0; r < (selected ? 0 : a.R); ++r) {
    Sel best{0u, 0xffffffffu, 0xffffffffu};
    if (LPT > 0) {
#pragma unroll
      for (int j = 0; j < kRegs; ++j) {
        if (key[j] == 0u || (best.key != 0u && key[j] < best.key)) continue;
        const int i = tid + j * kRerankThreads;
        const Sel s{key[j], uid_at(i), static_cast<uint32_t>(i)};
        if (best.key == 0u || sel_before(s, best)) best = s;
      }
    } else {
      if (r == 0) __syncthreads();  // bitmap cleared
      for (int i = tid; i < a.ncand; i += kRerankThreads) {
        if (retired[i >> 5] & (1u << (i & 31))) continue;
        const Sel s{order_key(cv[i]), uid_at(i), static_cast<uint32_t>(i)};
        if (s.key != 0u && (best.key == 0u || sel_before(s, best))) best = s;
      }
    }
    const Sel wb = warp_best(best);
    if (lane == 0) wbest[warp] = wb;
    __syncthreads();
    if (warp == 0) {
      const Sel fb = warp_best(wbest[lane]);
      if (lane == 0) {
        *chosen = fb;
        sel_id[r] = static_cast<int32_t>(fb.uid ^ 0x80000000u);
        if (LPT == 0 && fb.key != 0u) retired[fb.idx >> 5] |= 1u << (fb.idx & 31);
      }
    }
    __syncthreads();
    const uint32_t cidx = chosen->idx;
    if (LPT > 0) {
#pragma unroll
      for (int j = 0; j < kRegs; ++j)
        if (static_cast<uint32_t>(tid + j * kRerankThreads) == cidx) key[j] = 0u;
    }
  }
  __syncthreads();

  // exact rerank: wpr warps per selected row, each over a contiguous K range; the partial sums
  // are added in a fixed order
  int wpr = 1;
  while (wpr * 2 * a.R <= kRerankWarps && wpr < 8) wpr *= 2;
  const int k8_per = (a.K / 8 + wpr - 1) / wpr;
  for (int jw = warp; jw < a.R * wpr; jw += kRerankWarps) {
    const int j = jw / wpr, part = jw - j * wpr;
    const int n = sel_id[j];
    float logit = -INFINITY;
    if (n >= 0 && n < a.N) {
      const uint4* xr = reinterpret_cast<const uint4*>(xs);
      float acc = 0.0f;
      const int k8_end = min(a.K / 8, (part + 1) * k8_per);
      // kRerankUnroll loads of the weight row (16 bytes of bf16 or 8 of e4m3 each) in flight
      // per lane before any is used
      for (int k8b = part * k8_per + lane; k8b < k8_end; k8b += 32 * kRerankUnroll) {
        typename Row8<FP8>::Raw w8[kRerankUnroll];
#pragma unroll
        for (int u = 0; u < kRerankUnroll; ++u) {
          const int k8 = k8b + 32 * u;
          w8[u] = load_w8<FP8>(a, n, k8 < k8_end ? k8 : part * k8_per);
        }
#pragma unroll
        for (int u = 0; u < kRerankUnroll; ++u) {
          const int k8 = k8b + 32 * u;
          if (k8 < k8_end) {
            const uint4 x8 = xr[k8];
            const uint32_t xv[4] = {x8.x, x8.y, x8.z, x8.w};
            float part = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float wl, wh;
              w_pair(w8[u], q, wl, wh);
              part = fmaf(__uint_as_float(xv[q] << 16), wl, part);
              part = fmaf(__uint_as_float(xv[q] & 0xffff0000u), wh, part);
            }
            acc += part;
          }
        }
      }
      acc *= row_scale<FP8>(a, n);
#pragma unroll
      for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      logit = acc;
    } else if (n >= a.N && lane == 0 && part == 0) {
      set_status(a.status, DH_DEV_BAD_ID);
    }
    if (lane == 0) part_logit[jw] = logit;
  }
  __syncthreads();
  for (int j = tid; j < a.R; j += kRerankThreads) {
    float v = part_logit[j * wpr];
    for (int q = 1; q < wpr; ++q) v += part_logit[j * wpr + q];
    sel_logit[j] = v;
  }
  __syncthreads();

  if (warp == 0) {
    uint32_t bk = 0u, bu = 0xffffffffu;
    for (int j = lane; j < a.R; j += 32) {
      const uint32_t k = order_key(sel_logit[j]);
      const uint32_t u = static_cast<uint32_t>(sel_id[j]) ^ 0x80000000u;
      if (k > bk || (k == bk && u < bu)) {
        bk = k;
        bu = u;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t umin = __reduce_min_sync(0xffffffffu, bk == kmax ? bu : 0xffffffffu);
    if (lane == 0) {
      a.argmax_id[m] = static_cast<int32_t>(umin ^ 0x80000000u);
      if (a.h_argmax_id) a.h_argmax_id[m] = static_cast<int32_t>(umin ^ 0x80000000u);
    }
  }
  for (int j = tid; j < a.R; j += kRerankThreads) {
    a.rr_id[static_cast<int64_t>(m) * a.R + j] = sel_id[j];
    a.rr_logit[static_cast<int64_t>(m) * a.R + j] = sel_logit[j];
    if (a.h_rr_id) {
      a.h_rr_id[static_cast<int64_t>(m) * a.R + j] = sel_id[j];
      a.h_rr_logit[static_cast<int64_t>(m) * a.R + j] = sel_logit[j];
    }
    const int n = sel_id[j];
    if (a.y && n >= 0 && n < a.N)
      a.y[static_cast<int64_t>(m) * a.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sel_logit[j]));
  }
}



// ---- Cluster path (R <= 32, ncand <= 16384): one cluster of kRC CTAs per hidden row. The CTAs
// split the row's candidate slots and coordinate through distributed shared memory (no global
// round trips between phases, three cluster barriers); each computes R / kRC of the exact dots:
//  1. every CTA loads its slots (keys and ids in registers) and its copy of x, and sends its warp
//     maxima to every CTA of the cluster;
//  2. every CTA takes T = the R-th largest of the kRC * 8 warp maxima (a lower bound of the R-th
//     largest candidate, as in the single-CTA kernel) and writes its candidates with key >= T
//     into its own region of every CTA's survivor list;
//  3. every CTA selects the R first survivors in the selection order (the same ids everywhere;
//     or, if a region overflowed, runs the exact R-round selection over the whole row);
//  4. CTA r computes the dots of slots r, r + kRC, ...; CTA 0 takes the argmax.
constexpr int kRC = 8;
constexpr int kRCThreads = 256;
constexpr int kRCWarps = kRCThreads / 32;
constexpr int kRCMaxLPT = 8;
constexpr int kRCRegion = 64;  // survivors one CTA may place in each CTA's list
constexpr int kRCMaxR = 32;
constexpr int kRCMaxCand = kRC * kRCThreads * kRCMaxLPT;  // 16384

struct RCShared {
  uint32_t allmax[kRC * kRCWarps];  // the warp maxima of the cluster
  uint32_t T;                       // threshold
  int wcnt[kRCWarps];
  int rcnt[kRC];                    // survivors each CTA placed here (may exceed kRCRegion)
  Sel surv[kRC * kRCRegion];        // survivors, region r from CTA r
  Sel wbest[kRCWarps + 1];          // slow path
  int32_t rr[kRCMaxR];              // selected ids
  float part[4][kRCWarps];          // dot partials per warp, up to 4 slots per CTA
  float logit[kRCMaxR];             // CTA 0: reranked logits
  uint32_t retired[kRCMaxCand / 32];  // slow path: retired slots
};

template <typename T>
__device__ __forceinline__ T* cta0(cg::cluster_group& cl, T* p) {
  return cl.map_shared_rank(p, 0);
}

template <int LPT, bool FP8>
__global__ void __cluster_dims__(kRC, 1, 1) __launch_bounds__(kRCThreads, 1)
    rerank_cluster_kernel(const RerankArgs a) {
  cg::cluster_group cl = cg::this_cluster();
  __shared__ RCShared sh;
  const int rank = static_cast<int>(cl.block_rank());
  const int m = blockIdx.x / kRC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = (a.ncand + kRC - 1) / kRC;
  const int s0 = rank * chunk, s1 = min(a.ncand, s0 + chunk);
  const float* cv = a.cand_val + static_cast<int64_t>(m) * a.ncand;
  const int32_t* ci = a.cand_id + static_cast<int64_t>(m) * a.ncand;
  // the next kernel in the stream (the next call's coarse pass) may start its weight prefetch
  // on the SMs this small grid leaves idle; it waits for this grid before reading anything else
  if (tid == 0) grid_launch_dependents();

  // 1. once the preceding kernel has completed and its writes are visible (programmatic
  // dependent launch; a no-op otherwise): the keys and ids of this CTA's slots. x, which the dots
  // read straight from global memory (it may be that kernel's output), is only fetched into L2
  // before the wait.
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(m) * a.K);
  if (tid < a.K / 64) prefetch_l2(xr + 8 * tid);
  grid_dependency_wait();
  uint32_t key[LPT], uid[LPT];
#pragma unroll
  for (int j = 0; j < LPT; ++j) {
    const int i = s0 + tid + j * kRCThreads;
    key[j] = i < s1 ? order_key(cv[i]) : 0u;
    uid[j] = i < s1 ? static_cast<uint32_t>(ci[i]) ^ 0x80000000u : 0xffffffffu;
  }
  uint32_t tmax = 0u;
#pragma unroll
  for (int j = 0; j < LPT; ++j) tmax = max(tmax, key[j]);
  tmax = __reduce_max_sync(0xffffffffu, tmax);
  // every CTA receives every warp maximum (lane r writes CTA r's copy)
  if (lane < kRC) cl.map_shared_rank(sh.allmax, lane)[rank * kRCWarps + warp] = tmax;
  cl.sync();

  // 2. T: the R-th largest warp maximum (rank of each value by counting, ties by position), the
  // same in every CTA; then this CTA's candidates with key >= T into its region of every CTA
  if (warp == 0) {
    const uint32_t v0 = sh.allmax[lane], v1 = sh.allmax[32 + lane];
    int r0 = 0, r1 = 0;
    for (int src = 0; src < 32; ++src) {
      const uint32_t o0 = __shfl_sync(0xffffffffu, v0, src);
      const uint32_t o1 = __shfl_sync(0xffffffffu, v1, src);
      r0 += (o0 > v0 || (o0 == v0 && src < lane)) + (o1 > v0);
      r1 += (o0 >= v1) + (o1 > v1 || (o1 == v1 && src < lane));
    }
    const uint32_t T = __reduce_max_sync(
        0xffffffffu, max(r0 == a.R - 1 ? v0 : 0u, r1 == a.R - 1 ? v1 : 0u));
    if (lane == 0) sh.T = T;
  }
  __syncthreads();
  {
    const uint32_t T = sh.T;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < LPT; ++j) cnt += (key[j] != 0u && key[j] >= T) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sh.wcnt[warp] = incl;
    __syncthreads();
    int pos = incl - cnt, tot = 0;
    for (int w = 0; w < kRCWarps; ++w) {
      if (w < warp) pos += sh.wcnt[w];
      tot += sh.wcnt[w];
    }
#pragma unroll
    for (int j = 0; j < LPT; ++j)
      if (key[j] != 0u && key[j] >= T) {
        if (pos < kRCRegion) {
          const Sel v{key[j], uid[j], static_cast<uint32_t>(s0 + tid + j * kRCThreads)};
          for (int c = 0; c < kRC; ++c) cl.map_shared_rank(sh.surv, c)[rank * kRCRegion + pos] = v;
        }
        ++pos;
      }
    if (tid < kRC) cl.map_shared_rank(sh.rcnt, tid)[rank] = tot;
  }
  cl.sync();

  // 3. every CTA: the R first survivors in selection order (identical lists, identical ids)
  {
    int total = 0;
    bool overflow = false;
    for (int c = 0; c < kRC; ++c) {
      total += sh.rcnt[c];
      overflow = overflow || sh.rcnt[c] > kRCRegion;
    }
    if (!overflow) {
      if (warp == 0) {
        if (total <= 32) {
          Sel v{0u, 0xffffffffu, 0xffffffffu};
          if (lane < total) {
            int c = 0, l = lane;
            while (l >= sh.rcnt[c]) {
              l -= sh.rcnt[c];
              ++c;
            }
            v = sh.surv[c * kRCRegion + l];
          }
          v = warp_sort(v);
          if (lane < a.R) sh.rr[lane] = v.key ? static_cast<int32_t>(v.uid ^ 0x80000000u) : -1;
        } else {
          for (int r = 0; r < a.R; ++r) {
            Sel best{0u, 0xffffffffu, 0xffffffffu};
            for (int c = 0; c < kRC; ++c)
              for (int q = lane; q < sh.rcnt[c]; q += 32) {
                const Sel v = sh.surv[c * kRCRegion + q];
                if (v.key != 0u && (best.key == 0u || sel_before(v, best))) best = v;
              }
            const Sel wb = warp_best(best);
            for (int c = 0; c < kRC; ++c)
              for (int q = lane; q < sh.rcnt[c]; q += 32)
                if (sh.surv[c * kRCRegion + q].key != 0u && sh.surv[c * kRCRegion + q].idx == wb.idx)
                  sh.surv[c * kRCRegion + q].key = 0u;
            __syncwarp();
            if (lane == 0) sh.rr[r] = wb.key ? static_cast<int32_t>(wb.uid ^ 0x80000000u) : -1;
          }
        }
      }
    } else {
      // heavy ties overflowed a region: the exact R-round selection over the whole row
      for (int i = tid; i < (a.ncand + 31) / 32; i += kRCThreads) sh.retired[i] = 0u;
      __syncthreads();
      for (int r = 0; r < a.R; ++r) {
        Sel best{0u, 0xffffffffu, 0xffffffffu};
        for (int i = tid; i < a.ncand; i += kRCThreads) {
          if (sh.retired[i >> 5] & (1u << (i & 31))) continue;
          const Sel v{order_key(cv[i]), static_cast<uint32_t>(ci[i]) ^ 0x80000000u,
                      static_cast<uint32_t>(i)};
          if (v.key != 0u && (best.key == 0u || sel_before(v, best))) best = v;
        }
        const Sel wb = warp_best(best);
        if (lane == 0) sh.wbest[warp] = wb;
        __syncthreads();
        if (warp == 0) {
          const Sel fb =
              warp_best(lane < kRCWarps ? sh.wbest[lane] : Sel{0u, 0xffffffffu, 0xffffffffu});
          if (lane == 0) {
            sh.rr[r] = fb.key ? static_cast<int32_t>(fb.uid ^ 0x80000000u) : -1;
            if (fb.key != 0u) sh.retired[fb.idx >> 5] |= 1u << (fb.idx & 31);
          }
        }
        __syncthreads();
      }
    }
    __syncthreads();
    if (rank == 0 && tid < a.R) {
      const int32_t id = sh.rr[tid];
      a.rr_id[static_cast<int64_t>(m) * a.R + tid] = id;
      if (a.h_rr_id) a.h_rr_id[static_cast<int64_t>(m) * a.R + tid] = id;
    }
  }

  // 4. exact dots of this CTA's slots (rank, rank + kRC, ...): all of a thread's weight loads
  // for all its slots are in flight together; fixed-order reductions
  {
    const int nslot = (a.R - rank + kRC - 1) / kRC;  // 0..4
    const int k8n = a.K / 8;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int rown[4];
    bool live[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int n = u < nslot ? sh.rr[rank + u * kRC] : -1;
      live[u] = n >= 0 && n < a.N;
      rown[u] = live[u] ? n : 0;
    }
    for (int k8b = tid; k8b < k8n; k8b += kRCThreads * 3) {
      typename Row8<FP8>::Raw w8[4][3];
      uint4 xq[3];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int k8 = k8b + q * kRCThreads;
        xq[q] = k8 < k8n ? xr[k8] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const int k8 = k8b + q * kRCThreads;
          if (live[u] && k8 < k8n) w8[u][q] = load_w8<FP8>(a, rown[u], k8);
          else w8[u][q] = {};
        }
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int k8 = k8b + q * kRCThreads;
        if (k8 < k8n) {
          const uint4 x8 = xq[q];
          const uint32_t xv[4] = {x8.x, x8.y, x8.z, x8.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float p = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float wl, wh;
              w_pair(w8[u][q], e, wl, wh);
              p = fmaf(__uint_as_float(xv[e] << 16), wl, p);
              p = fmaf(__uint_as_float(xv[e] & 0xffff0000u), wh, p);
            }
            acc[u] += p;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] *= live[u] ? row_scale<FP8>(a, rown[u]) : 1.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int o = 16; o; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
      if (lane == 0) sh.part[u][warp] = acc[u];
    }
    __syncthreads();
    if (tid < nslot) {
      const int j = rank + tid * kRC;
      const int n = sh.rr[j];
      float v = -INFINITY;
      if (n >= 0 && n < a.N) {
        v = 0.0f;
        for (int w = 0; w < kRCWarps; ++w) v += sh.part[tid][w];
      } else if (n >= a.N) {
        set_status(a.status, DH_DEV_BAD_ID);
      }
      cta0(cl, sh.logit)[j] = v;
    }
  }
  cl.sync();

  // 5. CTA 0: outputs and the argmax (ties to the lowest id)
  if (rank == 0 && warp == 0) {
    uint32_t bk = 0u, bu = 0xffffffffu;
    for (int j = lane; j < a.R; j += 32) {
      const float v = sh.logit[j];
      const int32_t n = sh.rr[j];
      a.rr_logit[static_cast<int64_t>(m) * a.R + j] = v;
      if (a.h_rr_logit) a.h_rr_logit[static_cast<int64_t>(m) * a.R + j] = v;
      if (a.y && n >= 0 && n < a.N)
        a.y[static_cast<int64_t>(m) * a.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      const uint32_t k = order_key(v);
      const uint32_t u = static_cast<uint32_t>(n) ^ 0x80000000u;
      if (k > bk || (k == bk && u < bu)) {
        bk = k;
        bu = u;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t umin = __reduce_min_sync(0xffffffffu, bk == kmax ? bu : 0xffffffffu);
    if (lane == 0) {
      a.argmax_id[m] = static_cast<int32_t>(umin ^ 0x80000000u);
      if (a.h_argmax_id) a.h_argmax_id[m] = static_cast<int32_t>(umin ^ 0x80000000u);
    }
  }
}

template <int LPT, bool FP8>
static cudaError_t launch_rc(const RerankArgs& a, int M, cudaStream_t s) {
  const int smem = 0;
  cudaError_t e = cudaSuccess;
  // programmatic dependent launch: the CTAs may start (and fetch x into L2) while the kernel
  // before them in the stream finishes; they wait for its completion before reading anything
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M * kRC);
  cfg.blockDim = dim3(kRCThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, rerank_cluster_kernel<LPT, FP8>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int LPT, bool FP8>
static cudaError_t launch_rr(const RerankArgs& a, int M, cudaStream_t s) {
  size_t smem = static_cast<size_t>(2 * a.K) + sizeof(Sel) * (kRerankWarps + 1) +
                static_cast<size_t>(a.R) * 8 + static_cast<size_t>(a.R) * kRerankWarps * 4 +
                sizeof(Sel) * kSurvivorCap + 4 * (kRerankWarps + 2);
  if (LPT == 0) smem += 4 * static_cast<size_t>((a.ncand + 31) / 32);
  cudaError_t e = cudaFuncSetAttribute(rerank_argmax_kernel<LPT, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  rerank_argmax_kernel<LPT, FP8><<<M, kRerankThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <bool FP8>
static cudaError_t launch_rerank_fmt(const RerankArgs& a, const RerankCall& rc, cudaStream_t s) {
  const int M = static_cast<int>(rc.M);
  if (rc.R <= kRCMaxR && rc.ncand <= kRCMaxCand && rc.K <= 32768) {
    const int64_t lpt = ((rc.ncand + kRC - 1) / kRC + kRCThreads - 1) / kRCThreads;
    if (lpt <= 1) return launch_rc<1, FP8>(a, M, s);
    if (lpt <= 2) return launch_rc<2, FP8>(a, M, s);
    if (lpt <= 4) return launch_rc<4, FP8>(a, M, s);
    return launch_rc<8, FP8>(a, M, s);
  }
  const int64_t per = (rc.ncand + kRerankThreads - 1) / kRerankThreads;
  if (per <= 1) return launch_rr<1, FP8>(a, M, s);
  if (per <= 2) return launch_rr<2, FP8>(a, M, s);
  if (per <= 4) return launch_rr<4, FP8>(a, M, s);
  if (per <= 8) return launch_rr<8, FP8>(a, M, s);
  if (per <= 16) return launch_rr<16, FP8>(a, M, s);
  return launch_rr<0, FP8>(a, M, s);
}

cudaError_t launch_rerank_argmax(const RerankCall& rc, cudaStream_t s) {
  RerankArgs a{};
  a.x = static_cast<const uint16_t*>(rc.x);
  a.K = static_cast<int>(rc.K);
  a.N = static_cast<int>(rc.N);
  a.W = static_cast<const uint16_t*>(rc.W);
  a.W8 = rc.W8;
  a.wscale = rc.wscale;
  a.cand_val = rc.cand_val;
  a.cand_id = rc.cand_id;
  a.ncand = static_cast<int>(rc.ncand);
  a.R = rc.R;
  a.rr_id = rc.rr_id;
  a.rr_logit = rc.rr_logit;
  a.argmax_id = rc.argmax_id;
  a.y = static_cast<uint16_t*>(rc.y);
  a.status = rc.status;
  a.h_rr_id = rc.h_rr_id;
  a.h_rr_logit = rc.h_rr_logit;
  a.h_argmax_id = rc.h_argmax_id;
  return rc.W8 != nullptr ? launch_rerank_fmt<true>(a, rc, s) : launch_rerank_fmt<false>(a, rc, s);
}

}  // namespace dh
