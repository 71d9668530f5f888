// Coarse pass + block top-KCAND of the int2 draft head for many hidden rows at once (page
// "radiance_drafthead.py": module docstring, the int2 coarse kernel and the block candidate
// emission), on the
// 5th-generation tensor cores of sm_103a: tcgen05.mma with the dequantised weights in tensor
// memory (TMEM) and the hidden states in shared memory.
//
// Why only for many hidden rows: measured on GB300, one tcgen05.mma kind::f16 with M = 128,
// K = 16 occupies the tensor pipe for ~95 ns whatever N (16 .. 256) and wherever A comes from.
// Covering the vocabulary-scale head (124160 rows x 5120 codes) takes 310,400 such
// instructions, ~193 us on 152 SMs, for any number of hidden rows up to 256; the warp-level
// mma.sync kernel (coarse_kernel.cuh) takes 1/11 of that time per 16 x 16 tile step and wins
// while the hidden rows fit a few of its passes. Here one pass takes up to 80 hidden rows.
//
// Work decomposition:
//  * A prep kernel lays the pass's hidden states out as the MMA's B operand in the caller's
//    workspace: x * 2^(15 - E_m) as f16 (E_m from max |x[m]|), one contiguous unit per (scale
//    group J, plane p, quarter of the group's chunks); also the group sums XS and the E_m.
//  * Persistent grid, one CTA per SM, 128-row tiles (the MMA's M = TMEM lanes). One producer
//    thread feeds two rings without blocking on either: the packed rows through 128 x 128-byte
//    stages with 2-D tensor-map copies (TMA, 128-byte swizzle), and the B operand through
//    quarter slots (the four plane units of a quarter: four bulk copies, one barrier).
//  * 8 dequantising warps, two per TMEM lane quadrant (even and odd chunks); the thread of TMEM
//    lane r owns row r and, per tile, the exponent e of its largest scale (S 2^e in [8, 16)).
//    A 16-byte chunk of its row (16 byte positions x 4 planes) becomes 32 registers of f16
//    pairs: per word and plane one LOP3 puts the two codes c (times 4^p) into the mantissa of
//    1.0, and one HFMA2 with the pair (M, -M), M = S 2^(e + 10 - 2p), leaves exactly c S 2^e
//    (one rounding of a product with at most 10 significant bits). One tcgen05.st writes the
//    chunk's 32-column A stage: plane p's 16 codes are the stage's columns 8p .. 8p + 7.
//  * Three MMA-issuing threads (warps 1 .. 3): B quarter Q of the pass goes to issuer Q mod 3,
//    which accumulates all its quarters of the tile (every chunk and plane: the scale is in the
//    A operand) into its own D slot (128 x N fp32). A quarter's B slot and A stages belong to
//    its issuer alone: one wait for each and one commit releasing each per quarter, since one
//    thread issues an MMA only every ~100 ns and bookkeeping on that thread costs MMAs.
//  * 8 fold warps (two per TMEM lane quadrant, half of the columns each; thread = row) form the
//    zero-point part sum_g (S_g - ZS_g) XS_g while the tile's MMAs run, then add the three D
//    slots times 2^(E_m - e - 17), which is sum_g S_g sum x c / 4: together the page's
//    S (XS + sum x v / 4) - ZS XS summed over the groups. The tile's keys go to a per-CTA
//    column-major buffer in the workspace; the fold warps and 3 selection warps split the
//    top-KCAND of each 64-row block per hidden row (warp reductions on order-preserving keys,
//    lowest row on ties).
// Every wait is bounded (kWaitLimitNs); a wait that runs out marks the launch failed in the
// status word, after which every wait returns at once and the kernel runs to its end.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "dh_device.cuh"
#include "dh_launch.h"
#include "tc_device.cuh"

namespace dh {

constexpr int kWRows = 128;        // vocab rows per tile (MMA M, TMEM lanes)
constexpr int kWStageBytes = 128;  // packed bytes of a row per ring stage (8 chunks)
constexpr int kWStageSmem = kWRows * kWStageBytes;
constexpr int kWDeqWarps = 8;   // dequantising: two per TMEM lane quadrant
constexpr int kWFoldWarps = 8;  // fold: two per TMEM lane quadrant
constexpr int kWSelWarps = 3;   // block top-KCAND selection (off the critical path)
constexpr int kWSelWorkers = kWSelWarps + kWFoldWarps;  // the fold warps take a share too
constexpr int kWIssuers = 3;    // MMA-issuing threads: B quarter Q goes to issuer Q % 3
// warp 0: the copy producer (one thread, both rings); warps 1 .. 3: the MMA issuers; then the
// dequantising, fold and selection warps
constexpr int kWDeq0 = 1 + kWIssuers;          // first dequantising warp
constexpr int kWFold0 = kWDeq0 + kWDeqWarps;   // first fold warp
constexpr int kWSel0 = kWFold0 + kWFoldWarps;  // first selection warp
constexpr int kWWarps = kWSel0 + kWSelWarps;
constexpr int kWThreads = kWWarps * 32;
constexpr int kWMaxNP = 8;   // packed ring stages at most
constexpr int kWNB = 6;      // B ring slots: a quarter of a scale group each (four plane units)
constexpr int kWMaxGrid = 256;  // CTAs of a pass the per-CTA key buffers are sized for
constexpr int kWMaxNA = 14;  // A stages at most (32 TMEM columns each)
constexpr int kWTmemCols = 512;
constexpr int kWPrepThreads = 256;

struct WideArgs {
  int R;  // hidden rows of this pass (<= the MMA's N)
  int K, N, RB, KG, NJ, NC, NS, ntiles;
  const uint16_t* S;   // bf16 [N, KG]
  const uint16_t* ZS;  // bf16 [N, KG]
  const unsigned char* bbuf;  // B units [NJ][4][CPJ][2][NCOL][16 bytes] (prep)
  const float* xs;            // [NCOL][KG] group sums of x (prep)
  const int* ew;              // [NCOL] E_m (prep)
  int m0;                     // first hidden row of the pass (outputs)
  int kcand, nblk;
  float* cand_val;  // [M, nblk * kcand]
  int32_t* cand_id;
  uint16_t* y;  // bf16 [M, N] or nullptr
  uint32_t* status;
  int np, unit_bytes, szp;
  uint32_t* keys_g;  // per-CTA key buffers [grid][128][NCOL] (scratch)
  int off_bring, off_sz, off_xs, off_ew, off_bars;
};

__device__ __forceinline__ void w_cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ float w_pow2(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// ---- prep: one CTA per MMA column m (hidden row m0 + m of the pass; zeros past R) -------------
template <int G>
__global__ void __launch_bounds__(kWPrepThreads) wide_prep_kernel(const uint16_t* x, int m0,
                                                                  int R, int K, int ncol,
                                                                  unsigned char* bbuf, float* xs,
                                                                  int* ew) {
  // x may be an output of the preceding kernel, and the buffers may still be read by it (the
  // previous pass): wait for its completion before anything else
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  constexpr int CPJ = G / 16;
  __shared__ uint32_t red[kWPrepThreads / 32];
  const int m = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool live = m < R;
  const int RB = K / 4, KG = K / G;
  const uint16_t* xr = x + static_cast<int64_t>(m0 + (live ? m : 0)) * K;
  uint32_t mx = 0u;  // max |x| as bf16 magnitude bits
  if (live) {
    for (int i = tid; i < K / 8; i += kWPrepThreads) {
      const uint4 v = reinterpret_cast<const uint4*>(xr)[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = 0u;
#pragma unroll
  for (int i = 0; i < kWPrepThreads / 32; ++i) mx = max(mx, red[i]);
  int e = static_cast<int>(mx >> 7) - 126;  // max |x| = f 2^e, f in [0.5, 1)
  e = e < -100 ? -100 : (e > 100 ? 100 : e);
  if (tid == 0) ew[m] = live ? e : 0;
  // item it = ((J * 4 + p) * CPJ + cj) * 2 + h: the 8 values of K-half h of chunk c = J CPJ + cj
  // of plane p, in the order of the A columns (bytes 0, 2, 1, 3 of each word)
  for (int it = tid; it < K / 8; it += kWPrepThreads) {
    const int h = it & 1, t = it >> 1, cj = t % CPJ, t2 = t / CPJ, p = t2 & 3, J = t2 >> 2;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (live) {
      const int k0 = p * RB + 16 * (J * CPJ + cj) + 8 * h;
      const uint4 v = *reinterpret_cast<const uint4*>(xr + k0);
      const float sx = w_pow2(15 - e);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t hv[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        hv[2 * j] = __half_as_ushort(__float2half_rn(bf16_bits_to_float(w[j] & 0xffffu) * sx));
        hv[2 * j + 1] = __half_as_ushort(__float2half_rn(bf16_bits_to_float(w[j] >> 16) * sx));
      }
      out.x = hv[0] | (hv[2] << 16);
      out.y = hv[1] | (hv[3] << 16);
      out.z = hv[4] | (hv[6] << 16);
      out.w = hv[5] | (hv[7] << 16);
    }
    *reinterpret_cast<uint4*>(bbuf + (static_cast<int64_t>(it) * ncol + m) * 16) = out;
  }
  // group sums XS[m][g] (fixed order: lanes, then a butterfly)
  for (int gi = warp; gi < KG; gi += kWPrepThreads / 32) {
    float s = 0.0f;
    if (live)
      for (int i = lane; i < G; i += 32) s += bf16_bits_to_float(xr[gi * G + i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) xs[m * KG + gi] = s;
  }
}

// ---- the pass: NCOL = MMA N (16 .. 80), the pass's hidden rows in columns 0 .. R-1 -------------
template <int G, int NCOL>
__global__ void __launch_bounds__(kWThreads, 1)
    coarse_wide_kernel(const __grid_constant__ CUtensorMap tmap, const WideArgs a) {
  constexpr int P = 4;                       // int2 planes
  constexpr int CPJ = G / 16;                // chunks per scale group
  constexpr int CPQ = CPJ / 4;               // chunks per B quarter-unit
  constexpr int ACOLS = 32;                  // TMEM columns of one A stage: one chunk, four planes
  // kWIssuers D slots (one per issuer, a whole tile each) at columns 0 .. kWIssuers NCOL, then the
  // A stages, an even number (the two dequantising parities own alternate stages)
  constexpr int NAS = ((kWTmemCols - kWIssuers * NCOL) / ACOLS > kWMaxNA
                           ? kWMaxNA
                           : (kWTmemCols - kWIssuers * NCOL) / ACOLS) &
                      ~1;
  constexpr int NAQ = NAS / CPQ;  // A ring in quarters (the issuers' unit of work)
  constexpr int PITCH = NCOL;  // key buffer: [NCOL][128] words per CTA
  constexpr int HC = NCOL / 2;     // D columns of one fold warp
  static_assert(NCOL % 16 == 0 && NCOL >= 16 && NCOL <= 80, "MMA N");
  static_assert(NAS >= 2, "TMEM budget: at least one A stage per dequantising parity");
  static_assert(NAS % CPQ == 0 && NAQ >= 2, "A ring: whole quarters, at least two");
  static_assert(CPQ >= 1 && CPJ == 4 * CPQ, "four B quarter-units per (group, plane)");
  extern __shared__ unsigned char sm_raw[];
  // 1024-byte alignment for the 128-byte swizzle of the packed ring
  unsigned char* sm = sm_raw + ((1024u - (smem_addr(sm_raw) & 1023u)) & 1023u);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int np = a.np;
  uint64_t* pfull = reinterpret_cast<uint64_t*>(sm + a.off_bars);  // [kWMaxNP] stage landed
  uint64_t* pempty = pfull + kWMaxNP;   // [kWMaxNP] stage read by the dequantising warps
  uint64_t* bfull = pempty + kWMaxNP;   // [kWNB] B quarter landed (four plane units)
  uint64_t* bempty = bfull + kWNB;      // [kWNB] the quarter's issuer past it
  uint64_t* afull = bempty + kWNB;      // [NAQ used] a quarter's A stages written
  uint64_t* aempty = afull + kWMaxNA;   // [NAQ used] ... and its MMAs done
  uint64_t* dfull = aempty + kWMaxNA;   // the tile's D slots complete
  uint64_t* dempty = dfull + 1;         // ... and read by the fold warps
  uint64_t* mma_done = dempty + 1;      // every MMA of the CTA complete
  uint64_t* keys_ready = mma_done + 1;  // a tile's keys written by the fold warps
  uint64_t* keys_free = mma_done + 2;   // ... and consumed by the selection warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int my_tiles =
      (a.ntiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
      static_cast<int>(gridDim.x);
  const int total_stages = my_tiles * a.NS;
  const int quarters_per_tile = a.NJ * 4;  // B quarters of a tile: 4 per group

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWMaxNP; ++i) {
      mbar_init(&pfull[i], 1u);
      mbar_init(&pempty[i], static_cast<uint32_t>(kWDeqWarps));
    }
    for (int i = 0; i < kWNB; ++i) {
      mbar_init(&bfull[i], 1u);
      mbar_init(&bempty[i], 1u);  // the quarter's issuer
    }
    for (int i = 0; i < kWMaxNA; ++i) {
      mbar_init(&afull[i], 4u * CPQ);  // the quadrant warps of the quarter's chunks
      mbar_init(&aempty[i], 1u);        // the quarter's issuer
    }
    mbar_init(dfull, static_cast<uint32_t>(kWIssuers));
    mbar_init(dempty, static_cast<uint32_t>(kWFoldWarps));
    mbar_init(mma_done, static_cast<uint32_t>(kWIssuers));
    mbar_init(keys_ready, static_cast<uint32_t>(kWFoldWarps));
    mbar_init(keys_free, static_cast<uint32_t>(kWSelWorkers));
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_map(&tmap);
  }
  if (warp == 0) tmem_alloc(tmem_slot, kWTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_base = tmem + kWIssuers * NCOL;  // column of A stage 0 (D slot q at q NCOL)

  // Bounded wait on one phase of an mbarrier: one test first (the common case costs one
  // instruction and no clock read), then suspended waits. Returns at once (false) once the launch
  // is aborted; a wait that runs out aborts it. Callers go on either way (uniform control flow).
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
      if (*abort_flag) return false;
      if (mbar_try_wait(bar, parity)) return true;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        set_status(a.status, DH_DEV_WAIT_TIMEOUT);
        return false;
      }
    }
  };
  auto tile_of = [&](int lt) {
    return static_cast<int>(blockIdx.x) + lt * static_cast<int>(gridDim.x);
  };
  // ring position (slot, phase parity) advanced by one without a division
  auto advance = [](int& slot, uint32_t& ph, int n) {
    if (++slot == n) {
      slot = 0;
      ph ^= 1u;
    }
  };
  // the row's scale exponent: S 2^e in [8, 16) for the row's largest S (bf16 magnitude bits)
  auto scale_exponent = [](uint32_t max_bits) {
    return max_bits ? 130 - static_cast<int>(max_bits >> 7) : 0;
  };

  // block top-KCAND of this worker's share of a tile's jobs (job j = (64-row block j / R of the
  // tile, hidden row j % R)), from the tile's keys [NCOL][128]; a warp runs JB jobs at once so
  // that their warp reductions overlap (each round of one job is a chain of two)
  auto select_jobs = [&](int worker, int tile, const uint32_t* keys) {
    constexpr int JB = 4;
    for (int j0 = worker * JB; j0 < 2 * a.R; j0 += kWSelWorkers * JB) {
      uint32_t k0[JB], k1[JB], key_lo[JB], row_lo[JB], key_hi[JB], row_hi[JB];
      int bb[JB], mm[JB];
#pragma unroll
      for (int u = 0; u < JB; ++u) {
        const int jj = j0 + u;
        const int blk = jj / a.R;
        mm[u] = jj - blk * a.R;
        bb[u] = tile * 2 + blk;
        const bool live = jj < 2 * a.R && bb[u] < a.nblk;
        const uint32_t* kc = keys + mm[u] * kWRows + 64 * blk;
        k0[u] = live ? __ldcg(kc + lane) : 0u;  // L2: this CTA wrote them just before
        k1[u] = live ? __ldcg(kc + lane + 32) : 0u;
        key_lo[u] = key_hi[u] = 0u;  // slots lane, lane + 32
        row_lo[u] = row_hi[u] = 64u;
        if (!live) bb[u] = -1;
      }
      for (int r = 0; r < a.kcand; ++r) {
        uint32_t bk[JB], brow[JB], kmax[JB], rwin[JB];
#pragma unroll
        for (int u = 0; u < JB; ++u) {
          const bool first = k0[u] >= k1[u];
          bk[u] = first ? k0[u] : k1[u];
          brow[u] = first ? static_cast<uint32_t>(lane) : static_cast<uint32_t>(lane + 32);
          kmax[u] = __reduce_max_sync(0xffffffffu, bk[u]);
        }
#pragma unroll
        for (int u = 0; u < JB; ++u)
          rwin[u] = __reduce_min_sync(0xffffffffu, bk[u] == kmax[u] ? brow[u] : 64u);
#pragma unroll
        for (int u = 0; u < JB; ++u) {
          if (kmax[u] != 0u && lane == static_cast<int>(rwin[u] & 31u)) {
            if (rwin[u] < 32u) k0[u] = 0u; else k1[u] = 0u;
          }
          if (lane == (r & 31)) {
            if (r < 32) {
              key_lo[u] = kmax[u];
              row_lo[u] = kmax[u] ? rwin[u] : 64u;
            } else {
              key_hi[u] = kmax[u];
              row_hi[u] = kmax[u] ? rwin[u] : 64u;
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < JB; ++u) {
        if (bb[u] < 0) continue;
        const int b = bb[u];
        const int64_t obase = static_cast<int64_t>(a.m0 + mm[u]) * a.nblk * a.kcand +
                              static_cast<int64_t>(b) * a.kcand;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int slot = lane + 32 * h;
          const uint32_t kk = h ? key_hi[u] : key_lo[u], rr = h ? row_hi[u] : row_lo[u];
          if (slot < a.kcand) {
            a.cand_val[obase + slot] = kk ? key_to_float(kk) : -INFINITY;
            a.cand_id[obase + slot] = kk ? b * 64 + static_cast<int>(rr) : -1;
          }
        }
      }
    }
  };

  int issued = 0, issued_b = 0;  // copies issued into the packed and B rings (warp 0, lane 0)
  if (warp == 0) {
    // ---- one producer thread for both rings, in one fixed order: packed stage gs + np - 1,
    // then the B quarters of stage gs. Every wait is a suspended, bounded mbarrier wait (no
    // polling: the thread shares its SMSP with a dequantising warp). The order cannot deadlock:
    // a packed slot comes back once the dequantising warps finish stage gs - 1, whose A stages
    // need only MMAs on B quarters already issued; a B slot comes back once its issuer passes a
    // quarter six back, whose A stages need only packed stages already issued. The first packed
    // stages go to L2 while the preceding kernel may still run (it may have written the weights:
    // only L2, which is coherent, is touched before griddepcontrol.wait); every copy into shared
    // memory comes after the wait.
    if (lane == 0) {
      for (int s = 0; s < np && s < total_stages; ++s)
        tma_prefetch_l2_2d(&tmap, (s % a.NS) * kWStageBytes, tile_of(s / a.NS) * kWRows);
      grid_dependency_wait();
      constexpr int kQPS = 8 / CPQ;  // B quarters per packed stage (a stage is 8 chunks)
      int pslot = 0, bslot = 0, bunit = 0, p_st = 0, p_lt = 0;
      uint32_t pph = 0u, bph = 0u;
      // step gs issues packed stage gs + np - 1 and then stage gs's B quarters (steps before 0
      // only fill the packed ring)
      for (int gs = 1 - np; gs < total_stages && !*abort_flag; ++gs) {
        if (issued < total_stages) {
          if (issued >= np) wait_bar(&pempty[pslot], pph ^ 1u);
          if (*abort_flag) break;
          mbar_arrive_expect_tx(&pfull[pslot], static_cast<uint32_t>(kWStageSmem));
          tma_load_2d(sm + pslot * kWStageSmem, &tmap, p_st * kWStageBytes,
                      tile_of(p_lt) * kWRows, &pfull[pslot]);
          advance(pslot, pph, np);
          if (++p_st == a.NS) {
            p_st = 0;
            ++p_lt;
          }
          ++issued;
        }
        if (gs < 0) continue;
        for (int k = 0; k < kQPS && !*abort_flag; ++k) {
          if (issued_b >= kWNB) wait_bar(&bempty[bslot], bph ^ 1u);
          if (*abort_flag) break;
          // quarter (J, uq): the prep layout is (J, plane, chunk), so the quarter is four
          // contiguous plane units, one copy each, landing side by side in the slot
          const int uj = bunit >> 2, uq = bunit & 3;
          mbar_arrive_expect_tx(&bfull[bslot], static_cast<uint32_t>(P * a.unit_bytes));
#pragma unroll
          for (int up = 0; up < P; ++up)
            bulk_g2s(sm + a.off_bring + (bslot * P + up) * a.unit_bytes,
                     a.bbuf + static_cast<int64_t>((uj * 4 + up) * 4 + uq) * a.unit_bytes,
                     static_cast<uint32_t>(a.unit_bytes), &bfull[bslot]);
          advance(bslot, bph, kWNB);
          if (++bunit == quarters_per_tile) bunit = 0;
          ++issued_b;
        }
      }
    }
    __syncwarp();
  } else if (warp <= kWIssuers) {
    // ---- MMA issue: issuer q = warp - 1 takes the B quarters Q == q (mod 3) of the pass, all
    // chunks and planes of each (the scale is in the A operand, so every plane and group of the
    // tile accumulates into the issuer's one D slot). A B slot (Q mod 6) and an A quarter slot
    // always belong to one issuer, which alone waits for and releases them.
    const int q = warp - 1;
    if (lane == 0) {
      const uint32_t idesc = tc_idesc_f16(kWRows, NCOL);
      const uint64_t bdesc0 = tc_sdesc(smem_addr(sm + a.off_bring), NCOL * 16, 128u);
      const uint32_t d = tmem + q * NCOL;
      int aq = 0, bslot = 0;
      uint32_t aph = 0u, bph = 0u;
      int rq = 0;  // quarter index of the pass mod 3
      for (int lt = 0; lt < my_tiles; ++lt) {
        if (lt > 0) wait_bar(dempty, static_cast<uint32_t>(lt - 1) & 1u);
        bool first = true;  // the issuer's first MMA of the tile starts its D slot
        for (int J = 0; J < a.NJ; ++J) {
          for (int qq = 0; qq < 4; ++qq) {
            if (rq == q) {
              wait_bar(&bfull[bslot], bph);  // the quarter's four plane units
              wait_bar(&afull[aq], aph);     // its chunks' A stages
              tc_fence_after();
#pragma unroll
              for (int cc = 0; cc < CPQ; ++cc) {
#pragma unroll
                for (int p = 0; p < P; ++p) {
                  const uint64_t bd =
                      bdesc0 + static_cast<uint64_t>(
                                   ((bslot * P + p) * a.unit_bytes + cc * 2 * NCOL * 16) >> 4);
                  tc_mma_f16_ts(d, a_base + (aq * CPQ + cc) * ACOLS + 8 * p, bd, idesc,
                                !(first && cc == 0 && p == 0));
                }
              }
              first = false;
              tc_commit(&aempty[aq]);
              tc_commit(&bempty[bslot]);
            }
            advance(aq, aph, NAQ);
            advance(bslot, bph, kWNB);
            if (++rq == kWIssuers) rq = 0;
          }
        }
        tc_commit(dfull);
      }
      tc_commit(mma_done);
      mbar_wait_bounded(mma_done, 0u);  // also after an abort: no MMA may outlive the TMEM
    }
    __syncwarp();
  } else if (warp < kWFold0) {
    // ---- dequantisation: eight warps, two per TMEM lane quadrant (one for the even chunks, one
    // for the odd), one thread per row. A stage holds one chunk's four planes (32 columns) of 16
    // byte positions as f16 pairs c S 2^e: per pair one LOP3 puts the two codes (times 4^p) into
    // the mantissa of 1.0, one HFMA2 with the group's multiplier M = S 2^(e + 10 - 2p) and -M
    // leaves exactly c S 2^e (the FMA rounds once, and the product has at most 10 significant
    // bits) whenever S 2^e >= 2^-17, i.e. for every scale of at least 2^-20 of the row's largest;
    // below that it is off by less than one f16 subnormal step.
    const int sub = (warp - kWDeq0) >> 2;  // chunk parity of this warp
    const int row = (warp & 3) * 32 + lane;
    const uint32_t my_a = a_base + tmem_lane_base(warp);
    const int sw = row & 7;
    int ps = 0;  // packed ring slot of the current stage
    uint32_t pph = 0u;
    int as = sub;  // A ring slot of this warp's next chunk (the parities alternate: NAS is even)
    uint32_t aph = 0u;
    int done0 = 0;  // chunks of the pass before the current group
    grid_dependency_wait();  // the scales may be the preceding kernel's output (the quantiser)
    for (int lt = 0; lt < my_tiles; ++lt) {
      const int n = tile_of(lt) * kWRows + row;
      const uint16_t* srow = a.S + static_cast<int64_t>(n < a.N ? n : 0) * a.KG;
      if (lt + 1 < my_tiles) {  // the next tile's scale row heads for L2
        const int n1 = tile_of(lt + 1) * kWRows + row;
        if (n1 < a.N)
          prefetch_l2_bulk(a.S + static_cast<int64_t>(n1) * a.KG, static_cast<uint32_t>(a.KG * 2));
      }
      // the row's largest S: every 16-byte load of the row in flight together (K/G <= 80)
      uint32_t mx = 0u;
      {
        uint4 v[10];
#pragma unroll
        for (int i = 0; i < 10; ++i)
          v[i] = i < a.KG / 8 ? reinterpret_cast<const uint4*>(srow)[i] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < 10; ++i) {
          const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
        }
      }
      const int en = scale_exponent(mx);
      // the four planes' S of a group, loaded one group ahead
      uint32_t snext[P];
#pragma unroll
      for (int p = 0; p < P; ++p) snext[p] = srow[p * a.NJ];
      for (int J = 0; J < a.NJ; ++J) {
        const int c0 = J * CPJ;  // the group's first chunk within the tile
        // plane p's multiplier pair (M, -M) as f16x2
        uint32_t mul[P], bias[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const float sv = bf16_bits_to_float(snext[p]) * w_pow2(en + 10 - 2 * p);
          const uint32_t hm = __half_as_ushort(__float2half_rn(sv));
          mul[p] = hm | (hm << 16);
          bias[p] = mul[p] ^ 0x80008000u;
        }
        if (J + 1 < a.NJ) {
#pragma unroll
          for (int p = 0; p < P; ++p) snext[p] = srow[p * a.NJ + J + 1];
        }
        if ((c0 & 7) == 0) {  // the group starts a packed stage (8 chunks)
          wait_bar(&pfull[ps], pph);
          __syncwarp();
        }
        const unsigned char* prow = sm + ps * kWStageSmem + row * kWStageBytes;
        for (int cj = sub; cj < CPJ; cj += 2) {
          const int c = c0 + cj;
          const uint4 w4 = *reinterpret_cast<const uint4*>(prow + ((((c & 7) ^ sw)) << 4));
          const uint32_t t[4] = {w4.x, w4.y, w4.z, w4.w};
          uint32_t r[32];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t te = t[w], to = t[w] >> 8;
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const uint32_t mk = 0x00030003u << (2 * p);
              r[8 * p + 2 * w] = (te & mk) | 0x3C003C00u;
              r[8 * p + 2 * w + 1] = (to & mk) | 0x3C003C00u;
            }
          }
#pragma unroll
          for (int p = 0; p < P; ++p) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __half2 h = __hfma2(*reinterpret_cast<const __half2*>(&r[8 * p + i]),
                                        *reinterpret_cast<const __half2*>(&mul[p]),
                                        *reinterpret_cast<const __half2*>(&bias[p]));
              r[8 * p + i] = *reinterpret_cast<const uint32_t*>(&h);
            }
          }
          if (done0 + cj >= NAS) {  // the stage's previous MMAs are done
            wait_bar(&aempty[as / CPQ], aph ^ 1u);
            __syncwarp();
          }
          tc_fence_after();
          tmem_st_x32(my_a + as * ACOLS, r);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&afull[as / CPQ]);
          as += 2;
          if (as >= NAS) {
            as -= NAS;
            aph ^= 1u;
          }
        }
        done0 += CPJ;
        if (((c0 + CPJ) & 7) == 0) {  // the packed stage's last group: release it
          __syncwarp();
          if (lane == 0) mbar_arrive(&pempty[ps]);
          advance(ps, pph, np);
        }
      }
    }
  } else if (warp < kWSel0) {
    // ---- fold: two warps per TMEM lane quadrant, each NCOL/2 columns of its 32 rows. While the
    // tile's MMAs run, the zero-point part sum_g (S_g - ZS_g) XS_g; then the three D slots
    // (sum_g S_g sum x v times 2^(e + 15 - E_m)) in logit units added to it.
    const int fw = warp - kWFold0;  // 0..7
    const int half = fw >> 2;
    const int row = (warp & 3) * 32 + lane;
    const int col0 = half * HC;
    const uint32_t my_d = tmem + tmem_lane_base(warp) + col0;
    unsigned char* s_row = sm + a.off_sz + row * a.szp;  // this row's S ...
    unsigned char* z_row = s_row + kWRows * a.szp;       // ... and ZS
    // this CTA's key buffer [128][PITCH] in global memory (L2): written here, read by the
    // selection warps through L2
    uint32_t* keys = a.keys_g + static_cast<int64_t>(blockIdx.x) * kWRows * PITCH;
    float* xsd = reinterpret_cast<float*>(sm + a.off_xs);           // [KG][NCOL]
    int* ew_s = reinterpret_cast<int*>(sm + a.off_ew);              // [NCOL]
    // the half-0 warp copies the row's S, the half-1 warp its ZS; a barrier of the fold warps
    // then shares them
    auto load_sz = [&](int lt) {
      const int n = tile_of(lt) * kWRows + row;
      const bool valid = n < a.N;
      const int64_t off = static_cast<int64_t>(valid ? n : 0) * a.KG;
      const uint16_t* src = (half ? a.ZS : a.S) + off;
      unsigned char* dst = half ? z_row : s_row;
      for (int i = 0; i < a.KG / 8; ++i) w_cp_async16(smem_addr(dst + 16 * i), src + 8 * i, valid);
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // the first tile's scales into L2 while the preceding kernel may still run (only L2
    // before the wait, as for the packed rows); the copies into shared memory follow it
    if (my_tiles > 0) {
      const int n = tile_of(0) * kWRows + row;
      if (n < a.N)
        prefetch_l2_bulk((half ? a.ZS : a.S) + static_cast<int64_t>(n) * a.KG,
                         static_cast<uint32_t>(a.KG * 2));
    }
    // the prep kernel's group sums and exponents (the outputs are written after this wait too):
    // xsd[g][m] = XS[m][g]
    grid_dependency_wait();
    if (my_tiles > 0) load_sz(0);
    const int ftid = fw * 32 + lane;
    if (ftid < NCOL) ew_s[ftid] = a.ew[ftid];
    for (int i = ftid; i < NCOL * a.KG; i += kWFoldWarps * 32) {
      const int m = i / a.KG, gi = i - m * a.KG;
      xsd[gi * NCOL + m] = a.xs[i];
    }
    named_bar_sync(2, kWFoldWarps * 32);
    constexpr int kBatch = 8;  // D columns per load, three slots per wait
    for (int lt = 0; lt < my_tiles; ++lt) {
      const int n = tile_of(lt) * kWRows + row;
      const bool valid = n < a.N;
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      named_bar_sync(2, kWFoldWarps * 32);  // both halves' copies of the tile's S, ZS landed
      float acc[HC];
#pragma unroll
      for (int m = 0; m < HC; ++m) acc[m] = 0.0f;
      uint32_t mx = 0u;
      for (int gi = 0; gi < a.KG; ++gi) {
        const uint32_t sb = *reinterpret_cast<const uint16_t*>(s_row + 2 * gi);
        mx = max(mx, sb & 0x7fffu);
        const float zg = bf16_bits_to_float(sb) -
                         bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(z_row + 2 * gi));
        const float4* xg4 = reinterpret_cast<const float4*>(xsd + gi * NCOL + col0);
#pragma unroll
        for (int q = 0; q < HC; q += 4) {
          const float4 x4 = xg4[q >> 2];
          acc[q] = fmaf(zg, x4.x, acc[q]);
          acc[q + 1] = fmaf(zg, x4.y, acc[q + 1]);
          acc[q + 2] = fmaf(zg, x4.z, acc[q + 2]);
          acc[q + 3] = fmaf(zg, x4.w, acc[q + 3]);
        }
      }
      const int en = scale_exponent(mx);
      wait_bar(dfull, static_cast<uint32_t>(lt) & 1u);
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int q0 = 0; q0 < HC; q0 += kBatch) {
        uint32_t d0[kBatch], d1[kBatch], d2[kBatch];
        tmem_ld<8>(my_d + q0, d0);
        tmem_ld<8>(my_d + NCOL + q0, d1);
        tmem_ld<8>(my_d + 2 * NCOL + q0, d2);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const float dsum = (__uint_as_float(d0[i]) + __uint_as_float(d1[i])) +
                             __uint_as_float(d2[i]);
          acc[q0 + i] = fmaf(dsum, w_pow2(ew_s[col0 + q0 + i] - en - 17), acc[q0 + i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty);  // the D slots go back to the issuers
      named_bar_sync(2, kWFoldWarps * 32);  // both halves are done with the tile's S and ZS rows
      if (lt + 1 < my_tiles) load_sz(lt + 1);
      if (a.y != nullptr && valid) {
#pragma unroll
        for (int m = 0; m < HC; ++m)
          if (col0 + m < a.R)
            a.y[static_cast<int64_t>(a.m0 + col0 + m) * a.N + n] =
                __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
      }
      // hand the keys to the selection warps (a single buffer: wait until they are done with
      // the previous tile's)
      if (lt > 0) wait_bar(keys_free, static_cast<uint32_t>(lt - 1) & 1u);
      __syncwarp();
#pragma unroll
      for (int m = 0; m < HC; ++m) keys[(col0 + m) * kWRows + row] = valid ? order_key(acc[m]) : 0u;
      __syncwarp();
      if (lane == 0) mbar_arrive(keys_ready);
      // the fold warps are idle until the next tile's D slots fill: they take a share of the
      // tile's selection jobs once every fold warp's keys are written
      named_bar_sync(2, kWFoldWarps * 32);
      select_jobs(kWSelWarps + fw, tile_of(lt), keys);
      __syncwarp();
      if (lane == 0) mbar_arrive(keys_free);
    }
  } else {
    // ---- selection: block top-KCAND of every (64-row block, hidden row) of a tile -------------
    grid_dependency_wait();  // the outputs
    const int sw4 = warp - kWSel0;  // 0 .. kWSelWarps - 1
    const uint32_t* keys = a.keys_g + static_cast<int64_t>(blockIdx.x) * kWRows * PITCH;
    for (int lt = 0; lt < my_tiles; ++lt) {
      const int tile = tile_of(lt);
      wait_bar(keys_ready, static_cast<uint32_t>(lt) & 1u);
      __syncwarp();
      select_jobs(sw4, tile, keys);
      __syncwarp();
      if (lane == 0) mbar_arrive(keys_free);
    }
  }

  __syncthreads();
  if (warp == 0) {
    // after an abort, copies may still be in flight: they land before the CTA's shared memory
    // goes away
    if (lane == 0 && *abort_flag) {
      for (int ring = 0; ring < 2; ++ring) {
        const int n_iss = ring == 0 ? issued : issued_b, depth = ring == 0 ? np : kWNB;
        uint64_t* bars = ring == 0 ? pfull : bfull;
        for (int s = 0; s < depth && s < n_iss; ++s) {
          const int last = n_iss - 1 - ((n_iss - 1 - s) % depth);
          mbar_wait_bounded(&bars[s], static_cast<uint32_t>(last / depth) & 1u);
        }
      }
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kWTmemCols);
  }
}

// ---- host side ----------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static size_t round_up_sz(size_t v, size_t m) { return (v + m - 1) / m * m; }

size_t coarse_wide_scratch_bytes(int64_t M, int64_t K) {
  if (M <= kWideMinRows) return 0;
  const size_t kk = static_cast<size_t>(K);
  return round_up_sz(kWideMaxRows * kk * 2, 256) +          // B units
         round_up_sz(kWideMaxRows * (kk / 64) * 4, 256) +   // group sums (G >= 64)
         round_up_sz(kWideMaxRows * 4, 256) +               // exponents
         round_up_sz(static_cast<size_t>(kWMaxGrid) * kWRows * kWideMaxRows * 4, 256);  // keys
}

bool coarse_wide_supports(const CoarseCall& cc) {
  if (cc.bits != 2 || (cc.G != 64 && cc.G != 128) || cc.M <= kWideMinRows) return false;
  if (cc.K % 512 != 0 || (cc.K / cc.G) % 8 != 0 || cc.K / cc.G > 80) return false;
  return encode_tiled_fn() != nullptr;
}

// Shared-memory plan of a pass; false if the rings do not fit.
static bool plan_wide(WideArgs& a, int ncol, int G, int max_smem, int* smem_bytes) {
  const int cpj = G / 16;
  a.unit_bytes = (cpj / 4) * 2 * ncol * 16;  // a B quarter-unit
  a.szp = a.KG * 2;
  const int sz_bytes = 2 * kWRows * a.szp;
  const int xs_bytes = ncol * a.KG * 4;
  const int ew_bytes = ncol * 4;
  const int bar_bytes = (2 * kWMaxNP + 2 * kWNB + 2 * kWMaxNA + 2 + 3) * 8 + 16;
  const int fixed = sz_bytes + xs_bytes + ew_bytes + bar_bytes + 64 + 1024;  // keys: in the scratch
  // the B ring holds one and a half scale groups (kWNB quarters of four plane units)
  const int nbu = kWNB * 4;
  int np = (max_smem - fixed - nbu * a.unit_bytes) / kWStageSmem;
  if (np > kWMaxNP) np = kWMaxNP;
  if (np < 3) return false;
  a.np = np;
  a.off_bring = np * kWStageSmem;
  a.off_sz = a.off_bring + nbu * a.unit_bytes;
  a.off_xs = a.off_sz + sz_bytes;
  a.off_ew = a.off_xs + xs_bytes;
  a.off_bars = static_cast<int>(round_up_sz(a.off_ew + ew_bytes, 16));
  *smem_bytes = a.off_bars + bar_bytes + 1024;
  return *smem_bytes <= max_smem;
}

template <typename Kernel, typename... Args>
static cudaError_t launch_pdl(Kernel kernel, int grid, int threads, int smem, cudaStream_t s,
                              Args... args) {
  // programmatic dependent launch: the CTAs may start while the kernel before them in the
  // stream finishes; they wait for it (griddepcontrol.wait) before touching its outputs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int G, int NCOL>
static cudaError_t launch_wide_pass(const CUtensorMap& map, const WideArgs& a, int grid, int smem,
                                    const uint16_t* x, unsigned char* bbuf, float* xs, int* ew,
                                    cudaStream_t s) {
  cudaError_t e = launch_pdl(wide_prep_kernel<G>, NCOL, kWPrepThreads, 0, s, x, a.m0, a.R, a.K,
                             NCOL, bbuf, xs, ew);
  if (e != cudaSuccess) return e;
  auto kernel = coarse_wide_kernel<G, NCOL>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, grid, kWThreads, smem, s, map, a);
}

template <int G>
static cudaError_t launch_wide_g(int ncol, const CUtensorMap& map, const WideArgs& a, int grid,
                                 int smem, const uint16_t* x, unsigned char* bbuf, float* xs,
                                 int* ew, cudaStream_t s) {
  switch (ncol) {
    case 32: return launch_wide_pass<G, 32>(map, a, grid, smem, x, bbuf, xs, ew, s);
    case 48: return launch_wide_pass<G, 48>(map, a, grid, smem, x, bbuf, xs, ew, s);
    case 64: return launch_wide_pass<G, 64>(map, a, grid, smem, x, bbuf, xs, ew, s);
    default: return launch_wide_pass<G, 80>(map, a, grid, smem, x, bbuf, xs, ew, s);
  }
}

cudaError_t launch_coarse_wide(const CoarseCall& cc, void* scratch, int num_sms, int max_smem,
                               cudaStream_t s) {
  if (!coarse_wide_supports(cc) || scratch == nullptr) return cudaErrorNotSupported;
  WideArgs a{};
  a.K = static_cast<int>(cc.K);
  a.N = static_cast<int>(cc.N);
  a.RB = a.K / 4;
  a.KG = a.K / cc.G;
  a.NJ = a.RB / cc.G;
  a.NC = a.RB / 16;
  a.NS = a.RB / kWStageBytes;
  a.ntiles = (a.N + kWRows - 1) / kWRows;
  a.S = static_cast<const uint16_t*>(cc.S);
  a.ZS = static_cast<const uint16_t*>(cc.ZS);
  a.kcand = cc.kcand;
  a.nblk = static_cast<int>((cc.N + 63) / 64);
  a.cand_val = cc.cand_val;
  a.cand_id = cc.cand_id;
  a.y = static_cast<uint16_t*>(cc.y);
  a.status = cc.status;
  const size_t kk = static_cast<size_t>(cc.K);
  unsigned char* bbuf = static_cast<unsigned char*>(scratch);
  float* xs = reinterpret_cast<float*>(bbuf + round_up_sz(kWideMaxRows * kk * 2, 256));
  int* ew = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(xs) +
                                   round_up_sz(kWideMaxRows * (kk / 64) * 4, 256));
  a.bbuf = bbuf;
  a.xs = xs;
  a.ew = ew;
  a.keys_g = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(ew) +
                                         round_up_sz(kWideMaxRows * 4, 256));

  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.RB), static_cast<cuuint64_t>(a.N)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.RB)};
  const cuuint32_t box[2] = {kWStageBytes, kWRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode_tiled_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(cc.packed),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  int grid = a.ntiles < num_sms ? a.ntiles : num_sms;
  if (grid > kWMaxGrid) grid = kWMaxGrid;
  const int64_t passes = (cc.M + kWideMaxRows - 1) / kWideMaxRows;
  for (int64_t ps = 0; ps < passes; ++ps) {
    // rows spread evenly over the passes, each a multiple of 16 columns wide
    const int64_t m0 = ps * cc.M / passes, m1 = (ps + 1) * cc.M / passes;
    a.m0 = static_cast<int>(m0);
    a.R = static_cast<int>(m1 - m0);
    const int ncol = a.R <= 32 ? 32 : a.R <= 48 ? 48 : a.R <= 64 ? 64 : 80;
    int smem = 0;
    if (!plan_wide(a, ncol, cc.G, max_smem, &smem)) return cudaErrorInvalidValue;
    const cudaError_t e =
        cc.G == 128
            ? launch_wide_g<128>(ncol, map, a, grid, smem, static_cast<const uint16_t*>(cc.x),
                                 bbuf, xs, ew, s)
            : launch_wide_g<64>(ncol, map, a, grid, smem, static_cast<const uint16_t*>(cc.x),
                                bbuf, xs, ew, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dh
