// Coarse pass + block top-KCAND of the int2 draft head, up to 8 hidden rows per pass (page
// "radiance_drafthead.py": module docstring, and its int2 coarse-kernel and block-emit sections),
// for sm_103a. A warp-specialised streaming kernel:
//
//  * Persistent grid, one CTA per SM, walking 64-row candidate blocks b = blockIdx.x + j * grid;
//    each block is four 16-row tiles. NW = K / 256 MMA warps and three epilogue warps.
//  * The packed head streams in with ONE tensor-map copy per 16-row tile (TMA): a 3-D view of the
//    packed rows -- dim 0 the 64 bytes of a warp's strip, dim 1 the rows (stride K/4), dim 2 the
//    NW strips (stride 64) -- and a {64, 16, NW} box land the whole tile in the layout each MMA
//    warp reads, [warp][16 rows][64 bytes], into a ring of ns stages; rows past N come in as
//    zeros. There is no producer warp: the last MMA warp to release a stage (an arrival counter)
//    issues that stage's next copy, so no warp waits to refill the ring. Each block's S and ZS rows
//    (two bulk copies) come into a ring of nsb block stages the same way, refilled by the last
//    epilogue warp done with a block.
//  * MMA warp w owns the same 256 k-values of every vocab row (bytes [64w, 64w + 64) of each
//    packed row): its x fragments stay in registers for the whole launch. Per tile it checks the
//    stage, reads its strip (two 16-byte loads per lane, conflict-free), dequantises and
//    multiplies (below), folds the per-group scale into its accumulator, writes its partial sums
//    of the tile's rows and releases the stage. Nothing else: no copies to wait for, no epilogue.
//  * Dequant in place, as f16 subnormals: in an f16 pair every bit of the low byte of each half
//    is mantissa, so for a packed 32-bit word t the AND of t with plane p's code mask is the f16
//    pair (byte 0's code, byte 2's code) * 2^(2p - 24) exactly, and the same AND of t >> 8 gives
//    bytes 1 and 3: one logic op per MMA register (two weights). mma.sync m16n8k16, f16 in,
//    fp32 accumulate; weights on the 16-row side, hidden rows (or, for one hidden row, the four
//    scale groups of the strip) on the 8-column side.
//  * x enters the MMA as x * s / 4^p in f16 with s a power of two per (warp strip, hidden row)
//    (max |x s| in [2^14, 2^15)): exact for every element above max |x| * 2^-29.
//  * The page's dequant is 1 + v/4 with premultiplied S, ZS; a group contributes
//    S * (XS + sum x v / 4) - ZS * XS = S * sum x v / 4 + (S - ZS) * XS, so the MMA warps
//    accumulate S * sum x v (the scale on the accumulator, never on the weight tile) and the
//    zero-point part sum_g (S - ZS) XS is a short bf16 MMA chain per tile, run by the epilogue.
//  * The three epilogue warps take every block in order: they wait for its NW partial sets,
//    compute the zero-point part (split by tile, handed over through an mbarrier), then split the
//    hidden rows: each sums the partials of its rows in a fixed order (deterministic), selects the
//    block's top-KCAND with warp reductions (max key, lowest row on ties) and writes the
//    candidates. They poll with __nanosleep between tests, so that they take almost no issue slots
//    from the MMA warps; up to four partial buffers hide their wake-up latency.
// Every wait is bounded (kWaitLimitNs): a wait that runs out marks the launch failed in the status
// word and every later wait returns at once; thread 0 then waits (bounded) for the copies still in
// flight before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "dh_device.cuh"
#include "dh_launch.h"
#include "tc_device.cuh"

namespace dh {

namespace {

constexpr int kSMaxNW = 20;      // K <= 5120
constexpr int kEpi = 3;          // epilogue warps
constexpr int kSMaxRed = 4;      // partial buffers
constexpr int kSMaxThreads = (kSMaxNW + kEpi) * 32;
constexpr int kSMaxStages = 8;   // packed tile stages
constexpr int kSMaxSZ = 4;       // S/ZS block stages
constexpr int kStrip = 64;       // packed bytes of a warp's strip of one row
constexpr int kWarpTile = kTileRows * kStrip;  // 1 KB: one warp's part of a tile

// a bf16 of shared memory, as the low bits of a word
__device__ __forceinline__ uint32_t lds_bf16(const unsigned char* p) {
  return *reinterpret_cast<const uint16_t*>(p);
}
// Adds one to a shared-memory counter where `pred` holds and returns its previous value (0 where
// it does not), without a branch: the lanes that skip it do not wait for it.
__device__ __forceinline__ int atom_inc_if(int* p, bool pred) {
  int old;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\tmov.u32 %0, 0;\n\t"
      "@q atom.shared::cta.add.u32 %0, [%1], 1;\n\t}"
      : "=r"(old)
      : "r"(smem_addr(p)), "r"(pred ? 1u : 0u)
      : "memory");
  return old;
}
// One arrival on `bar` where `pred` holds (release at CTA scope), without a branch.
__device__ __forceinline__ void mbar_arrive_if(uint64_t* bar, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "@q mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_addr(bar)),
      "r"(pred ? 1u : 0u)
      : "memory");
}

struct StreamArgs {
  const uint16_t* x;  // bf16 [M, K]
  int M, m0, mt;      // this pass: hidden rows m0 .. m0 + mt - 1 (1 <= mt <= 8)
  int K, N, KG, NW;
  const uint16_t* S;   // bf16 [N, KG]
  const uint16_t* ZS;  // bf16 [N, KG]
  int kcand, nblk;
  float* cand_val;  // [M, nblk * kcand]
  int32_t* cand_id;
  uint16_t* y;  // bf16 [M, N] or nullptr
  uint32_t* status;
  uint32_t u16_mul;  // 2^16: bf16 bits -> fp32 as an integer multiply (FMA pipe, not ALU)
  int ns, nsb, nb, rp;  // tile stages, S/ZS stages, partial buffers, partial row pitch
  int off_bars, off_xs, off_zb, off_sz, off_red, off_zp, off_ring;
};

template <int G, int KSPEC, bool MT1>
__global__ void __launch_bounds__(kSMaxThreads, 1)
    coarse_stream_kernel(const __grid_constant__ CUtensorMap tmap, const StreamArgs a) {
  constexpr int P = 4;   // int2 planes
  constexpr int NQ = 4;  // scale groups of a strip (one per plane)
  extern __shared__ __align__(128) unsigned char sm[];
  const int K = KSPEC ? KSPEC : a.K;
  const int NW = K / 256, KG = KSPEC ? KSPEC / G : a.KG, RB = K / 4;
  const int mt = MT1 ? 1 : a.mt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int rp = MT1 ? 1 : a.rp;
  const int ns = a.ns, nsb = a.nsb, nb = a.nb;

  uint64_t* tile_full = reinterpret_cast<uint64_t*>(sm + a.off_bars);  // [kSMaxStages]
  uint64_t* sz_full = tile_full + kSMaxStages;                         // [kSMaxSZ]
  uint64_t* red_full = sz_full + kSMaxSZ;                              // [kSMaxRed]
  uint64_t* red_empty = red_full + kSMaxRed;                           // [kSMaxRed]
  uint64_t* zp_done = red_empty + kSMaxRed;                            // [kSMaxRed]
  int* tcnt = reinterpret_cast<int*>(zp_done + kSMaxRed);  // [kSMaxStages] releases of a stage
  int* tiss = tcnt + kSMaxStages;                          // [kSMaxStages] last tile issued
  int* scnt = tiss + kSMaxStages;                          // [kSMaxSZ] epilogue warps done
  int* siss = scnt + kSMaxSZ;                              // [kSMaxSZ] last block issued
  volatile int* abort_flag = siss + kSMaxSZ;
  float* xs_part = reinterpret_cast<float*>(sm + a.off_xs);  // [NW][8][NQ] strip group sums
  float* xs_full = xs_part + NW * 8 * NQ;                    // [mt][KG] group sums XS
  uint2* zb = reinterpret_cast<uint2*>(sm + a.off_zb);  // [KG/8][3][mt][4] zero-point B frags
  unsigned char* sz = sm + a.off_sz;                      // [nsb][S|ZS][64][KG] bf16
  float* red = reinterpret_cast<float*>(sm + a.off_red);  // [nb][NW][64][rp] partials
  float* zpb = reinterpret_cast<float*>(sm + a.off_zp);   // [nb][64][rp] zero-point parts
  unsigned char* ring = sm + a.off_ring;                  // [ns][NW][16][64] packed tiles
  const int sz_half = kBlockRows * KG * 2;
  const int tstage = NW * kWarpTile;
  const int red_wstride = kBlockRows * rp;

  const int my_blocks = (a.nblk - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                        static_cast<int>(gridDim.x);
  const int ntiles = kTilesPerBlock * my_blocks;
  auto block_row0 = [&](int lb) {
    return (static_cast<int>(blockIdx.x) + lb * static_cast<int>(gridDim.x)) * kBlockRows;
  };

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(a.status, DH_DEV_WAIT_TIMEOUT);
  };
  // Bounded wait of one thread: tests spaced by `sleep_ns` of __nanosleep (the abort flag and
  // the clock looked at every 64 tests), or with sleep_ns == 0 suspended waits (try_wait) with the
  // flag and the clock looked at after each. False once the launch is aborted (its
  // own timeout or another thread's).
  auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t sleep_ns) -> bool {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      // sleep_ns == 0: the hardware's suspended wait (woken by the phase's completion)
      if (sleep_ns ? mbar_test_wait(bar, parity) : mbar_try_wait_hw(bar, parity)) return true;
      if (sleep_ns) __nanosleep(sleep_ns);
      if (sleep_ns == 0u || (it & 63u) == 0u) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          fail();
          return false;
        }
      }
    }
  };
  // The same for a whole warp (every lane takes the same path: the loops hold warp-wide MMAs and
  // reductions). Fast path: every lane tests the phase itself and one vote says all saw it
  // complete; else lane 0 waits, the outcome is broadcast and every lane observes the phase.
  auto wait_warp = [&](uint64_t* bar, uint32_t parity, uint32_t sleep_ns) -> bool {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    int ok = 1;
    if (lane == 0) ok = wait1(bar, parity, sleep_ns) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_test_wait(bar, parity);
    return ok != 0;
  };
  // Tile tau of this CTA into ring stage s (one thread). A tile wholly past N (the head's last
  // block) is not copied: its phase completes at once and the MMA warps read stale codes for rows
  // the epilogue ignores.
  auto issue_tile = [&](int tau, int s) {
    tiss[s] = tau;
    const int row = block_row0(tau / kTilesPerBlock) + kTileRows * (tau % kTilesPerBlock);
    if (row < a.N) {
      mbar_arrive_expect_tx(&tile_full[s], static_cast<uint32_t>(tstage));
      tma_load_3d(ring + s * tstage, &tmap, 0, row, 0, &tile_full[s]);
    } else {
      mbar_arrive(&tile_full[s]);
    }
  };
  // S and ZS rows of local block lb into block stage st (one thread).
  auto issue_sz = [&](int lb, int st) {
    siss[st] = lb;
    const int row0 = block_row0(lb);
    const int rows = a.N - row0 > kBlockRows ? kBlockRows : a.N - row0;
    const uint32_t bytes = static_cast<uint32_t>(rows * KG * 2);  // KG % 8 == 0
    unsigned char* dst = sz + st * 2 * sz_half;
    mbar_arrive_expect_tx(&sz_full[st], 2u * bytes);
    bulk_g2s(dst, a.S + static_cast<int64_t>(row0) * KG, bytes, &sz_full[st]);
    bulk_g2s(dst + sz_half, a.ZS + static_cast<int64_t>(row0) * KG, bytes, &sz_full[st]);
  };

  if (threadIdx.x == 0) {
    for (int q = 0; q < kSMaxStages; ++q) {
      mbar_init(&tile_full[q], 1u);
      tcnt[q] = 0;
      tiss[q] = -1;
    }
    for (int q = 0; q < kSMaxSZ; ++q) {
      mbar_init(&sz_full[q], 1u);
      scnt[q] = 0;
      siss[q] = -1;
    }
    for (int q = 0; q < kSMaxRed; ++q) {
      mbar_init(&red_full[q], static_cast<uint32_t>(NW));
      mbar_init(&red_empty[q], static_cast<uint32_t>(kEpi));
      mbar_init(&zp_done[q], static_cast<uint32_t>(kEpi));
    }
    *abort_flag = 0;
    mbar_fence_init();
    // Before griddepcontrol.wait only L2 is warmed (the preceding kernel may have written the
    // weights; L2 is coherent): the first tiles and S/ZS stages.
    tma_prefetch_map(&tmap);
    for (int tau = 0; tau < ns && tau < ntiles; ++tau)
      tma_prefetch_l2_3d(&tmap, 0, block_row0(tau >> 2) + kTileRows * (tau & 3), 0);
    for (int lb = 0; lb < nsb && lb < my_blocks; ++lb) {
      const int row0 = block_row0(lb);
      const int rows = a.N - row0 > kBlockRows ? kBlockRows : a.N - row0;
      prefetch_l2_bulk(a.S + static_cast<int64_t>(row0) * KG, static_cast<uint32_t>(rows * KG * 2));
      prefetch_l2_bulk(a.ZS + static_cast<int64_t>(row0) * KG, static_cast<uint32_t>(rows * KG * 2));
    }
  }
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    for (int lb = 0; lb < nsb && lb < my_blocks; ++lb) issue_sz(lb, lb);
    for (int tau = 0; tau < ns && tau < ntiles; ++tau) issue_tile(tau, tau);
  }

  // ---- MMA warps: x fragments of the strip (B operand), strip sums of each scale group --------
  const int strip_byte = warp * kStrip;
  const bool mma_warp = warp < NW;
  constexpr int BP = MT1 ? 1 : P;
  uint32_t bfr[4][BP][2];
  int ew = 0;  // E of this warp's strip of the lane's hidden row (max |x| = f 2^E, f in [.5, 1))
  const int q_own = MT1 && g < NQ ? g : 0;  // MT1: this lane's scale group (= plane)
  if (mma_warp) {
    const int xrow = MT1 ? 0 : (g < mt ? g : 0);
    const bool xval = MT1 || g < mt;
    const uint16_t* xg = a.x + static_cast<int64_t>(a.m0 + xrow) * K;
    uint2 xv[4][P];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < P; ++p)
        xv[i][p] = xval ? *reinterpret_cast<const uint2*>(xg + p * (K / P) + strip_byte + 16 * c +
                                                          4 * i)
                        : make_uint2(0u, 0u);
    uint32_t mx = 0;
    float xsg[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) xsg[q] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const uint2 v = xv[i][p];
        mx = max(mx, max(max(v.x & 0x7fffu, (v.x >> 16) & 0x7fffu),
                         max(v.y & 0x7fffu, (v.y >> 16) & 0x7fffu)));
        xsg[p] += (bf16_bits_to_float(v.x & 0xffffu) + bf16_bits_to_float(v.x >> 16)) +
                  (bf16_bits_to_float(v.y & 0xffffu) + bf16_bits_to_float(v.y >> 16));
      }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));  // the row's four lanes
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      xsg[q] += __shfl_xor_sync(0xffffffffu, xsg[q], 1);
      xsg[q] += __shfl_xor_sync(0xffffffffu, xsg[q], 2);
    }
    ew = static_cast<int>(mx >> 7) - 126;
    ew = ew < -100 ? -100 : (ew > 100 ? 100 : ew);  // zero or tiny rows
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < BP; ++p) bfr[i][p][0] = bfr[i][p][1] = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const float sx = __uint_as_float(static_cast<uint32_t>(15 - ew - 2 * p + 127) << 23);
        const uint2 v = xv[i][p];
        const uint32_t h[4] = {v.x & 0xffffu, v.x >> 16, v.y & 0xffffu, v.y >> 16};
        uint32_t hs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          hs[e] = __half_as_ushort(__float2half_rn(bf16_bits_to_float(h[e]) * sx));
        const uint32_t r0 = hs[0] | (hs[2] << 16);  // (x[k0], x[k0+2]): even bytes of the word
        const uint32_t r1 = hs[1] | (hs[3] << 16);  // (x[k0+1], x[k0+3]): odd bytes
        if (MT1) {
          if (p == q_own) {
            bfr[i][0][0] = r0;
            bfr[i][0][1] = r1;
          }
        } else {
          bfr[i][MT1 ? 0 : p][0] = r0;
          bfr[i][MT1 ? 0 : p][1] = r1;
        }
      }
    if (c == 0 && g < mt) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) xs_part[(warp * 8 + g) * NQ + q] = xsg[q];
    }
  }
  __syncthreads();  // barriers initialised, strip sums published
  // a dependent kernel (the rerank) may be scheduled as SMs free up; it waits for this grid's
  // completion before it reads anything this kernel writes
  if (threadIdx.x == 0) grid_launch_dependents();
  {
    const int RBG = RB / G;  // groups per plane
    for (int e = threadIdx.x; e < mt * KG; e += blockDim.x) {
      const int m = e / KG, col = e - m * KG;
      const int p = col / RBG, r0 = (col - p * RBG) * G;  // plane, first byte of the group
      float sum = 0.0f;
      for (int w = r0 / kStrip; w <= (r0 + G - 1) / kStrip; ++w) sum += xs_part[(w * 8 + m) * NQ + p];
      xs_full[m * KG + col] = sum;
    }
  }
  __syncthreads();
  // B fragments of the zero-point MMA: k' < KG is +XS[k'] (against S), KG <= k' < 2KG is
  // -XS[k' - KG] (against ZS); each value split exactly into bf16 hi + mid + lo.
  for (int e = threadIdx.x; e < (KG / 8) * 3 * mt * 4; e += blockDim.x) {
    const int cc = e & 3, m = (e >> 2) % mt, kp = (e >> 2) / mt;  // kp = kk * 3 + part
    const int kk = kp / 3, part = kp - kk * 3;
    uint32_t r[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t hv[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int kq = 16 * kk + 8 * h + 2 * cc + j;
        float v = kq < KG ? xs_full[m * KG + kq] : -xs_full[m * KG + kq - KG];
        float pv = 0.0f;
        for (int q = 0; q <= part; ++q) {
          pv = __bfloat162float(__float2bfloat16_rn(v));
          v -= pv;  // exact: v and pv share the leading bits
        }
        hv[j] = __bfloat16_as_ushort(__float2bfloat16_rn(pv));
      }
      r[h] = hv[0] | (hv[1] << 16);
    }
    zb[e] = make_uint2(r[0], r[1]);
  }
  __syncthreads();

  if (warp >= NW) {
    // ---- epilogue warps e = 0 .. kEpi - 1: every block, in order; warp e computes the zero point
    // of tiles e, e + kEpi, ... and then selects for hidden rows e, e + kEpi, ...
    const int e = warp - NW;
    int buf = 0, ph = 0;
    for (int lb = 0; lb < my_blocks; ++lb) {
      if (!wait_warp(&red_full[buf], static_cast<uint32_t>(ph), 128u)) break;
      const int st = lb % nsb;
      const unsigned char* stage = sz + st * 2 * sz_half;
      // the stage's copies landed before the MMA warps' arrivals; observe their phase here too
      // (it cannot move on before the epilogue releases the stage)
      mbar_test_wait(&sz_full[st], static_cast<uint32_t>(lb / nsb) & 1u);
      float* zp = zpb + buf * kBlockRows * rp;
      const float* rbuf = red + buf * NW * red_wstride;
      // zero-point part of the block, per 16-row tile: A = [S | ZS] rows (bf16, as stored),
      // B = [XS ; -XS] in three bf16 parts; D rows g, g + 8 x hidden rows 2c, 2c + 1
      {
        const uint2* zl = zb + (g < mt ? g : 0) * 4 + c;
        const bool zlive = g < mt;
        const int row8 = 8 * KG * 2;
#pragma unroll 1
        for (int t = e; t < kTilesPerBlock; t += kEpi) {
          // three independent chains (the hi, mid and lo parts of XS), added in a fixed order
          float zq[3][4] = {};
          const unsigned char* srow = stage + (t * kTileRows + g) * KG * 2 + 4 * c;
          for (int kk = 0; kk < KG / 8; ++kk) {
            uint32_t av[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int o8 = 16 * kk + 8 * h;  // first column of the octet (all S or all ZS)
              const unsigned char* src = o8 < KG ? srow + 2 * o8 : srow + sz_half + 2 * (o8 - KG);
              av[2 * h] = *reinterpret_cast<const uint32_t*>(src);
              av[2 * h + 1] = *reinterpret_cast<const uint32_t*>(src + row8);
            }
#pragma unroll
            for (int part = 0; part < 3; ++part) {
              const uint2 b = zlive ? zl[(kk * 3 + part) * mt * 4] : make_uint2(0u, 0u);
              mma_bf16_16816_acc(zq[part], av[0], av[1], av[2], av[3], b.x, b.y);
            }
          }
          float z[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) z[j] = (zq[0][j] + zq[1][j]) + zq[2][j];
          float* zw = zp + (t * kTileRows + g) * rp;
          if (2 * c < mt) {
            zw[2 * c] = z[0];
            zw[8 * rp + 2 * c] = z[2];
          }
          if (2 * c + 1 < mt) {
            zw[2 * c + 1] = z[1];
            zw[8 * rp + 2 * c + 1] = z[3];
          }
        }
      }
      // every epilogue warp's tiles of the zero point are written
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        mbar_arrive(&zp_done[buf]);
      }
      if (!wait_warp(&zp_done[buf], static_cast<uint32_t>(ph), 0u)) break;
      const int b = static_cast<int>(blockIdx.x) + lb * static_cast<int>(gridDim.x);
      const int n0 = b * kBlockRows + lane;
      for (int m = e; m < mt; m += kEpi) {
        float v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // fixed summation order (deterministic): four interleaved chains, then pairwise
          const float* rb = rbuf + (lane + 32 * h) * rp + m;
          float s0 = zp[(lane + 32 * h) * rp + m], s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
          int w = 0;
          for (; w + 4 <= NW; w += 4) {
            s0 += rb[w * red_wstride];
            s1 += rb[(w + 1) * red_wstride];
            s2 += rb[(w + 2) * red_wstride];
            s3 += rb[(w + 3) * red_wstride];
          }
          for (; w < NW; ++w) s0 += rb[w * red_wstride];
          v[h] = (s0 + s1) + (s2 + s3);
        }
        if (a.y) {
          uint16_t* yr = a.y + static_cast<int64_t>(a.m0 + m) * a.N;
          if (n0 < a.N) yr[n0] = __bfloat16_as_ushort(__float2bfloat16_rn(v[0]));
          if (n0 + 32 < a.N) yr[n0 + 32] = __bfloat16_as_ushort(__float2bfloat16_rn(v[1]));
        }
        uint32_t k0 = n0 < a.N ? order_key(v[0]) : 0u;
        uint32_t k1 = n0 + 32 < a.N ? order_key(v[1]) : 0u;
        uint32_t key_lo = 0u, row_lo = 64u, key_hi = 0u, row_hi = 64u;  // slots lane, lane + 32
        for (int r = 0; r < a.kcand; ++r) {
          const bool first = k0 >= k1;
          const uint32_t bk = first ? k0 : k1;
          const uint32_t brow = first ? static_cast<uint32_t>(lane) : static_cast<uint32_t>(lane + 32);
          const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
          const uint32_t rwin = __reduce_min_sync(0xffffffffu, bk == kmax ? brow : 64u);
          if (kmax != 0u && lane == static_cast<int>(rwin & 31u)) {
            if (rwin < 32u) k0 = 0u; else k1 = 0u;
          }
          if (lane == (r & 31)) {
            if (r < 32) {
              key_lo = kmax;
              row_lo = kmax ? rwin : 64u;
            } else {
              key_hi = kmax;
              row_hi = kmax ? rwin : 64u;
            }
          }
        }
        const int64_t obase = static_cast<int64_t>(a.m0 + m) * a.nblk * a.kcand +
                              static_cast<int64_t>(b) * a.kcand;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int slot = lane + 32 * h;
          const uint32_t kk = h ? key_hi : key_lo, rr = h ? row_hi : row_lo;
          if (slot < a.kcand) {
            a.cand_val[obase + slot] = kk ? key_to_float(kk) : -INFINITY;
            a.cand_id[obase + slot] = kk ? b * kBlockRows + static_cast<int>(rr) : -1;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        mbar_arrive(&red_empty[buf]);  // the partial buffer and the zero-point scratch
        // the S/ZS stage: the MMA warps were done with it before the block's partials were
        // complete; the last epilogue warp done with the block refills it
        if (atomicAdd(&scnt[st], 1) == kEpi - 1) {
          scnt[st] = 0;
          __threadfence_block();
          if (lb + nsb < my_blocks) {
            fence_proxy_async_smem();  // the stage's reads come before the copy's writes
            issue_sz(lb + nsb, st);
          }
        }
      }
      if (++buf == nb) { buf = 0; ph ^= 1; }
    }
  } else {
    // ---- MMA warps ---------------------------------------------------------------------------
    // S column of scale group q (= plane q) of this strip: q * (RB / G) + strip_byte / G
    const int so_g = g * KG * 2;
    const int row8 = 8 * KG * 2;
    // factor kappa / s that turns this lane's partials into logits: hidden rows 2c, 2c + 1
    // (MT1: the one hidden row, in ysc[0]); kappa = 2^24 / 4
    float ysc[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int hr = MT1 ? 0 : 2 * c + j, src = (hr < 8 ? hr : 0) * 4;
      const int e = __shfl_sync(0xffffffffu, ew, src);
      ysc[j] = hr < mt ? __uint_as_float(static_cast<uint32_t>(e + 7 + 127) << 23) : 0.0f;
    }
    // MT1: lane c folds groups 2c, 2c + 1 (lanes c >= 2 fold a valid group's scale into zero
    // columns: no effect)
    const int qa = MT1 ? (2 * c < NQ ? 2 * c : 0) : 0;
    auto s_col = [&](int q) { return q * (RB / G) + strip_byte / G; };
    const int soa = so_g + 2 * s_col(qa), sob = so_g + 2 * s_col(qa + 1 < NQ ? qa + 1 : qa);
    // Ring positions are fixed per block: ns is 4 or 8, so block lb's tiles sit in stages
    // s0 .. s0 + 3 with s0 = 4 (lb & 1) (ns = 8) or 0 (ns = 4), all of the same phase parity.
    // The release of a stage is lane 0's predicated counter add; whether this warp was the last
    // of the NW (and so refills the stage) is looked at one tile later, when the add's result is
    // long back, by a warp vote: no lane waits on the add, and the warp never diverges for it.
    int st = 0, stph = 0, buf = 0, rph = 0;
    int pend_old = 0, pend_s = 0, pend_tau = -1;  // the last release: lane 0's counter value
    auto refill_if_last = [&]() {
      if (__any_sync(0xffffffffu, lane == 0 && pend_tau >= 0 && pend_old == NW - 1)) {
        if (lane == 0) {
          tcnt[pend_s] = 0;
          __threadfence_block();
          const int nxt = pend_tau + ns;
          if (nxt < ntiles) {
            fence_proxy_async_smem();  // the stage's reads come before the copy's writes
            issue_tile(nxt, pend_s);
          }
        }
        __syncwarp();
      }
    };
    for (int lb = 0; lb < my_blocks; ++lb) {
      bool ok = wait_warp(&sz_full[st], static_cast<uint32_t>(stph), 0u);
      if (ok && lb >= nb) ok = wait_warp(&red_empty[buf], static_cast<uint32_t>(rph ^ 1), 0u);
      if (!ok) break;
      const unsigned char* stage = sz + st * 2 * sz_half;
      float* rwb = red + buf * NW * red_wstride + warp * red_wstride + g * rp + (MT1 ? 0 : 2 * c);
      const int s0 = ns == 8 ? 4 * (lb & 1) : 0;
      const uint32_t tph = static_cast<uint32_t>(ns == 8 ? (lb >> 1) & 1 : lb & 1);
      const unsigned char* cs0 = ring + s0 * tstage + warp * kWarpTile;
      bool rdy = mbar_test_wait(&tile_full[s0], tph);
#pragma unroll
      for (int t = 0; t < kTilesPerBlock; ++t) {
        if (!__all_sync(0xffffffffu, rdy) && !wait_warp(&tile_full[s0 + t], tph, 0u)) {
          ok = false;
          break;
        }
        const unsigned char* cs = cs0 + t * tstage;
        const unsigned char* szs = stage + t * (kTileRows * KG * 2);
        const uint4 wa = *reinterpret_cast<const uint4*>(cs + g * kStrip + 16 * c);
        const uint4 wb = *reinterpret_cast<const uint4*>(cs + (g + 8) * kStrip + 16 * c);
        // the next tile's stage, tested now so that the answer is back when it is needed
        if (t + 1 < kTilesPerBlock) rdy = mbar_test_wait(&tile_full[s0 + t + 1], tph);
        const uint32_t ta[4] = {wa.x, wa.y, wa.z, wa.w}, tb[4] = {wb.x, wb.y, wb.z, wb.w};
        float* rw = rwb + t * kTileRows * rp;
        if (MT1) {
          // one accumulator per scale group q (four independent chains); column q of dq[q] is
          // group q's dot, the other columns are ignored
          float dq[NQ][4];
#pragma unroll
          for (int q = 0; q < NQ; ++q) dq[q][0] = dq[q][1] = dq[q][2] = dq[q][3] = 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t tao = ta[i] >> 8, tbo = tb[i] >> 8;
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const uint32_t mk = 0x00030003u << (2 * p);
              mma_f16_16816_acc(dq[p], ta[i] & mk, tb[i] & mk, tao & mk, tbo & mk, bfr[i][0][0],
                                bfr[i][0][1]);
            }
          }
          // lane c holds columns 2c, 2c + 1: group 2c in dq[2c][0, 2], group 2c + 1 in
          // dq[2c + 1][1, 3] (rows g, g + 8); groups 2, 3 sit in lane c = 1
          const bool hi = c & 1;
          const float da0 = hi ? dq[2][0] : dq[0][0];
          const float da2 = hi ? dq[2][2] : dq[0][2];
          const float db1 = hi ? dq[3][1] : dq[1][1];
          const float db3 = hi ? dq[3][3] : dq[1][3];
          const float sa = __uint_as_float(lds_bf16(szs + soa) * a.u16_mul);
          const float sb = __uint_as_float(lds_bf16(szs + sob) * a.u16_mul);
          const float sa8 = __uint_as_float(lds_bf16(szs + soa + row8) * a.u16_mul);
          const float sb8 = __uint_as_float(lds_bf16(szs + sob + row8) * a.u16_mul);
          float r0 = fmaf(sb, db1, sa * da0);
          float r8 = fmaf(sb8, db3, sa8 * da2);
          r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
          r8 += __shfl_xor_sync(0xffffffffu, r8, 1);
          // partials in logit units: rows g and g + 8, from lane c = 0
          const float v0 = r0 * ysc[0], v8 = r8 * ysc[0];
          if (c == 0) rw[0] = v0;
          if (c == 0) rw[8] = v8;
        } else {
          float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          uint32_t tao[4], tbo[4];  // odd bytes moved down: t >> 8
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            tao[i] = ta[i] >> 8;
            tbo[i] = tb[i] >> 8;
          }
          // plane by plane: the plane's accumulator is folded as soon as it is complete
#pragma unroll
          for (int p = 0; p < P; ++p) {
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const uint32_t mk = 0x00030003u << (2 * p);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma_f16_16816_acc(d, ta[i] & mk, tb[i] & mk, tao[i] & mk, tbo[i] & mk,
                                bfr[i][MT1 ? 0 : p][0], bfr[i][MT1 ? 0 : p][1]);
            const unsigned char* sq = szs + so_g + 2 * s_col(p);
            const float sg = __uint_as_float(lds_bf16(sq) * a.u16_mul);
            const float sg8 = __uint_as_float(lds_bf16(sq + row8) * a.u16_mul);
            acc[0] = fmaf(sg, d[0], acc[0]);
            acc[1] = fmaf(sg, d[1], acc[1]);
            acc[2] = fmaf(sg8, d[2], acc[2]);
            acc[3] = fmaf(sg8, d[3], acc[3]);
          }
          // partials in logit units, D layout: acc[0..1] = row g, hidden rows 2c, 2c + 1;
          // acc[2..3] = row g + 8
          const float v0 = acc[0] * ysc[0], v1 = acc[1] * ysc[1];
          const float v2 = acc[2] * ysc[0], v3 = acc[3] * ysc[1];
          const bool lo = 2 * c < mt, hi1 = 2 * c + 1 < mt;
          if (lo) rw[0] = v0;
          if (lo) rw[8 * rp] = v2;
          if (hi1) rw[1] = v1;
          if (hi1) rw[8 * rp + 1] = v3;
        }
        // the previous release's refill, if this warp was its last arriver
        refill_if_last();
        // this stage has been read (every lane's loads were consumed above): release it
        __syncwarp();
        pend_old = atom_inc_if(&tcnt[s0 + t], lane == 0);
        pend_s = s0 + t;
        pend_tau = kTilesPerBlock * lb + t;
      }
      if (!ok) break;
      // the block's partials are written: hand them to the epilogue (the arrival releases them)
      __syncwarp();
      mbar_arrive_if(&red_full[buf], lane == 0);
      // the block's last release is looked at now: a warp about to wait for the epilogue must not
      // hold back the ring
      refill_if_last();
      pend_tau = -1;
      if (++st == nsb) { st = 0; stph ^= 1; }
      if (++buf == nb) { buf = 0; rph ^= 1; }
    }
    refill_if_last();  // the last release (its next tile, if any, is another warp's to wait for)
  }
  __syncthreads();
  // After an abort, copies may still be in flight: they land before the CTA's shared memory goes
  // away (bounded waits on the last phase each stage was given; completed phases return at once).
  if (threadIdx.x == 0 && *abort_flag) {
    for (int q = 0; q < ns; ++q)
      if (tiss[q] >= 0) mbar_wait_bounded(&tile_full[q], static_cast<uint32_t>(tiss[q] / ns) & 1u);
    for (int q = 0; q < nsb; ++q)
      if (siss[q] >= 0) mbar_wait_bounded(&sz_full[q], static_cast<uint32_t>(siss[q] / nsb) & 1u);
  }
}

// ---- host side ----------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

int round16(int v) { return (v + 15) / 16 * 16; }

// Shared-memory plan of a pass of `mt` hidden rows: the deepest tile ring that fits, preferring
// two partial buffers and four S/ZS stages. False if nothing fits.
bool plan_stream(StreamArgs& a, int mt, int max_smem, int* smem) {
  const int NW = a.NW;
  a.rp = mt == 1 ? 1 : (mt | 1);  // odd: a warp reading one column over 32 rows hits 32 banks
  // {partial buffers, S/ZS stages, tile stages}
  // {partial buffers, S/ZS stages, tile stages}; the kernel takes 4 or 8 tile stages
  static const int kPlans[][3] = {{4, 4, 8}, {3, 4, 8}, {2, 4, 8}, {2, 2, 8}, {1, 4, 8},
                                  {2, 4, 4}, {2, 2, 4}, {1, 4, 4}, {1, 2, 4}};
  for (const auto& pl : kPlans) {
    const int nb = pl[0], nsb = pl[1], ns = pl[2];
    int off = 0;
    a.off_bars = off;
    off += (kSMaxStages + kSMaxSZ + 3 * kSMaxRed) * 8 + (2 * kSMaxStages + 2 * kSMaxSZ + 1) * 4;
    a.off_xs = off = round16(off);
    off += NW * 8 * 4 * 4 + mt * a.KG * 4;
    a.off_zb = off = round16(off);
    off += (a.KG / 8) * 3 * mt * 4 * 8;
    a.off_sz = off = (off + 127) / 128 * 128;
    off += nsb * 2 * kBlockRows * a.KG * 2;
    a.off_red = off = round16(off);
    off += nb * NW * kBlockRows * a.rp * 4;
    a.off_zp = off = round16(off);
    off += nb * kBlockRows * a.rp * 4;
    a.off_ring = off = (off + 127) / 128 * 128;
    off += ns * NW * kWarpTile;
    if (off <= max_smem) {
      a.nb = nb;
      a.nsb = nsb;
      a.ns = ns;
      *smem = off;
      return true;
    }
  }
  return false;
}

template <int G, int KS, bool M1>
cudaError_t launch_stream_kernel(const CUtensorMap& map, const StreamArgs& a, int grid, int smem,
                                 cudaStream_t s) {
  auto kernel = coarse_stream_kernel<G, KS, M1>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the CTAs may start (and warm L2) while the kernel before them
  // in the stream finishes; everything else waits for it (griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((a.NW + kEpi) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, map, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_stream_g(const CUtensorMap& map, const StreamArgs& a, int grid, int smem,
                            cudaStream_t s) {
  if (a.K == 5120)
    return a.mt == 1 ? launch_stream_kernel<G, 5120, true>(map, a, grid, smem, s)
                     : launch_stream_kernel<G, 5120, false>(map, a, grid, smem, s);
  return a.mt == 1 ? launch_stream_kernel<G, 0, true>(map, a, grid, smem, s)
                   : launch_stream_kernel<G, 0, false>(map, a, grid, smem, s);
}

}  // namespace

bool coarse_stream_supports(const CoarseCall& cc) {
  if (cc.bits != 2 || (cc.G != 64 && cc.G != 128)) return false;
  if (cc.K % 256 != 0 || cc.K / 256 > kSMaxNW || (cc.K / cc.G) % 8 != 0 || cc.K < 8 * cc.G)
    return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_coarse_stream(const CoarseCall& cc, int num_sms, int max_smem, cudaStream_t s) {
  if (!coarse_stream_supports(cc)) return cudaErrorNotSupported;
  StreamArgs a{};
  a.x = static_cast<const uint16_t*>(cc.x);
  a.M = static_cast<int>(cc.M);
  a.K = static_cast<int>(cc.K);
  a.N = static_cast<int>(cc.N);
  a.KG = a.K / cc.G;
  a.NW = a.K / 256;
  a.S = static_cast<const uint16_t*>(cc.S);
  a.ZS = static_cast<const uint16_t*>(cc.ZS);
  a.kcand = cc.kcand;
  a.nblk = static_cast<int>((cc.N + kBlockRows - 1) / kBlockRows);
  a.cand_val = cc.cand_val;
  a.cand_id = cc.cand_id;
  a.y = static_cast<uint16_t*>(cc.y);
  a.status = cc.status;
  a.u16_mul = 1u << 16;

  // the packed rows as a 3-D tensor: (64 bytes of a strip, row, strip); a {64, 16, NW} box is one
  // 16-row tile in the [strip][row][64 bytes] layout the MMA warps read
  CUtensorMap map;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kStrip), static_cast<cuuint64_t>(a.N),
                              static_cast<cuuint64_t>(a.NW)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.K / 4), static_cast<cuuint64_t>(kStrip)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kStrip), static_cast<cuuint32_t>(kTileRows),
                             static_cast<cuuint32_t>(a.NW)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (encode_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(cc.packed), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorNotSupported;

  // passes of 8 hidden rows, or fewer when their partial buffers do not fit
  int pass_rows = 8, smem = 0;
  for (; pass_rows >= 1; pass_rows /= 2) {
    const int mt = a.M < pass_rows ? a.M : pass_rows;
    if (plan_stream(a, mt, max_smem, &smem)) break;
  }
  if (pass_rows < 1) return cudaErrorNotSupported;
  const int grid = a.nblk < num_sms ? a.nblk : num_sms;
  for (int m0 = 0; m0 < a.M; m0 += pass_rows) {
    a.m0 = m0;
    a.mt = a.M - m0 < pass_rows ? a.M - m0 : pass_rows;
    if (!plan_stream(a, a.mt, max_smem, &smem)) return cudaErrorNotSupported;
    const cudaError_t e = cc.G == 128 ? launch_stream_g<128>(map, a, grid, smem, s)
                                      : launch_stream_g<64>(map, a, grid, smem, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dh
