// Coarse pass + block top-KCAND of the low-bit draft head (page "radiance_drafthead.py":
// module docstring, the int2 coarse kernel and the block candidate emission), for sm_103a.
//
// Work decomposition (GB300-first, not the page's one-program-per-block grid):
//  * Persistent grid, one CTA per SM. A CTA walks 64-row candidate blocks b = blockIdx.x,
//    blockIdx.x + gridDim.x, ...; each block is four 16-row tiles.
//  * NW = K/256 warps. Warp w owns the same 256 k-values of every vocab row (its "strip": bytes
//    [64w, 64w+64) of each int2 row, [128w, 128w+128) of each int4 row). So:
//      - its share of the hidden states never changes: the x fragments of the MMA's B operand
//        live in registers for the whole launch;
//      - it streams only its own strip of each tile (16 rows x 64 B) through a private ring of
//        shared-memory stages with 16-byte cp.async copies, NSW-1 tiles ahead: no warp waits for
//        another warp's weights.
//  * S and ZS of a block (64 contiguous rows each) arrive by two bulk (TMA) copies into a ring of
//    block stages. The last arrival at the end of block b (an arrival counter: every warp, plus
//    the zero-point pass) knows that every warp is done with b's stage and partials; it refills
//    the stage with the S and ZS of the block that
//    comes nsb (2 or 4) later and publishes b's epilogue as one job per hidden row. Warps claim jobs
//    at block boundaries and while they wait (so the fastest warps do them, in parallel): a job
//    sums the NW partials of its rows in a fixed order (deterministic), selects the top-KCAND
//    with warp reductions (max key, lowest row on ties) and writes the candidates; the block's
//    last job releases its partial buffer. A warp waits only when it runs nsb blocks ahead
//    of the slowest warp (S stage) or nb blocks ahead of the epilogues (partial buffers).
//  * Dequant in place, as f16 subnormals: in an f16 pair every bit of the low byte of each half
//    is mantissa, so for a packed 32-bit word t (bytes b0..b3) the AND of t with the plane's
//    code mask gives the f16 pair (b0's code, b2's code) * 2^(-24 + shift) exactly, and the
//    same AND of t >> 8 gives (b1's code, b3's code): one LOP3 per MMA register (two weights),
//    one shift per word. int2 planes 0..3 sit at bits 2p, 2p+1 (factor 2^(2p)); int4 nibbles at
//    bits 0-3 and 4-7 (factor 2^(4p)). mma.sync m16n8k16 (f16 in, fp32 accumulate): weights on
//    the 16-row side, hidden rows on the 8-column side; bytes j and j+2 of a word share an A
//    register, and x is permuted the same way.
//  * The hidden states enter the MMA's B operand as x * s / 2^shift in f16, with s a power of
//    two per hidden row (max |x * s| in [2^14, 2^15)): exact for every element above the f16
//    normal threshold, i.e. for all but those below max |x| * 2^-29 (error < 2^-25 scaled).
//  * The page's dequant is 1 + v/L (L = 4 for int2, 16 for int4) on the group's S and ZS: a group
//    contributes S * (XS + sum x v / L) - ZS * XS = S * sum x v / L + (S - ZS) * XS. With the MMA
//    result D = s * 2^-24 * sum x v per (plane, group) of the strip, the warp accumulates
//    acc = sum S * D and its partial of the row is (kappa / s) * acc, kappa = 2^24 / L (powers of
//    two, exact). The zero-point part Z = sum_g (S - ZS) * XS of a 16-row tile is one more short
//    MMA chain: A = the tile's S and ZS rows as they are (bf16, K/G + K/G columns), B = XS and
//    -XS split exactly into three bf16 parts (hi, mid, lo), fp32 accumulation. The first warp to
//    finish a block runs it for the block's four tiles and writes it to an extra partial slot,
//    so the per-tile loop has no zero-point work and no per-tile branch.
//  * One hidden row (M = 1): the MMA's 8 columns would be 7/8 idle, so each scale group q of the
//    strip gets its own column q. The lanes of B column g hold the x values of their own group
//    g only (8 registers instead of 32), every MMA of group q accumulates into its own
//    accumulator, and only column q of that accumulator is read (the others pair group q's
//    weights with another group's x and are ignored). The per-group scale is then applied once
//    per tile per group (lanes c = 0, 1 hold columns 0..3).
//  * The per-group scale is applied to the accumulator, never to the weight tile.
// Hidden rows are processed eight at a time (one MMA column tile); M > 8 runs ceil(M/8) passes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "dh_device.cuh"
#include "dh_launch.h"

namespace dh {

constexpr int kCoarseMaxWarps = 20;  // K <= 5120
constexpr int kCoarseMaxThreads = kCoarseMaxWarps * 32;
constexpr int kSBlocks = 4;     // S/ZS block stages at most (the plan picks 4 or 2)
constexpr int kMaxRedBufs = 4;  // partial buffers (blocks)

struct CoarseArgs {
  const uint16_t* x;  // bf16 [M, K]
  int M, m0, mt;      // this pass covers hidden rows m0 .. m0+mt-1 (1 <= mt <= 8)
  int K, N, G, KG, RB, NW;
  const uint8_t* packed;  // [N, RB]
  const uint16_t* S;      // [N, KG] bf16
  const uint16_t* ZS;     // [N, KG] bf16
  int kcand, nblk;
  float* cand_val;  // [M, nblk*kcand]
  int32_t* cand_id;
  uint16_t* y;  // bf16 [M, N] or nullptr
  uint32_t* status;
  // 2^16 (bf16 bits -> fp32): a kernel parameter, so that the conversion stays an integer
  // multiply on the FMA pipe instead of a shift on the ALU pipe, which the dequant's ANDs keep
  // busy. (The t >> 8 of the odd bytes is a shift: an integer multiply-high runs at a quarter of
  // the ALU rate and stalls the tensor pipe's MMAs.)
  uint32_t u16_mul;
  // shared-memory plan
  int nb, red_pitch, nsb, nsb_log;  // partial buffers, their row pitch, S/ZS stages (2^nsb_log)
  int off_bars, off_xs, off_zb, off_sz, off_red, off_ring;
};

// 16-byte copy global -> shared (shared-space address); valid = false copies zeros.
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_dst), "l"(gsrc),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t lds_u16(const unsigned char* p) {
  return *reinterpret_cast<const uint16_t*>(p);
}

// f16 weights (two per register) of plane p from a packed word: code mask of the plane.
template <int BITS>
__device__ __forceinline__ uint32_t dq16(uint32_t t, int p) {
  if (BITS == 2) return t & (0x00030003u << (2 * p));  // v * 2^(2p - 24)
  return t & (0x000F000Fu << (4 * p));                 // v * 2^(4p - 24)
}
// log2 of the factor 2^shift of plane p's weights; the plane's x goes in divided by it.
template <int BITS>
__host__ __device__ constexpr int plane_shift(int p) {
  return BITS == 2 ? 2 * p : 4 * p;
}

// G: the quantisation group (64 or 128). KSPEC: the hidden size K when it is known at compile
// time (the vocabulary-scale head), 0 for a runtime K: with K fixed, every shared-memory offset
// and stride below is an immediate. NSW: stages of each warp's private weight ring. MT1: a single
// hidden row in this pass (scale groups in the MMA's columns).
template <int BITS, int G, int KSPEC, int NSW, bool MT1>
__global__ void __launch_bounds__(kCoarseMaxThreads, 1) coarse_topk_kernel(const CoarseArgs a) {
  // SPLIT: the strip spans two quantisation groups per plane (int4 with G = 64), so the
  // accumulator is folded once per 64-byte sub-chunk instead of once per strip.
  constexpr bool SPLIT = BITS == 4 && G == 64;
  constexpr int P = 8 / BITS;             // codes per byte (planes)
  constexpr int SB = 256 / P;             // strip bytes per row: 256 k-values
  constexpr int U = SB / 64;              // 64-byte sub-chunks per strip
  constexpr int FS = SPLIT ? U : 1;       // fold segments per strip
  constexpr int NQ = FS * P;              // scale groups per strip (<= 4)
  constexpr int WSTAGE = kTileRows * SB;  // packed bytes of one warp's strip of a tile
  constexpr int CH = WSTAGE / 16 / 32;    // 16-byte weight copies per lane per tile
  constexpr int kLogL = BITS == 2 ? 2 : 4;  // log2 of the page's divisor L
  constexpr int KGS = KSPEC ? KSPEC / G : 0;  // K/G when K is compiled in
  static_assert((NSW & (NSW - 1)) == 0, "ring depth must be a power of two");
  static_assert(NQ <= 4, "scale groups of a strip must fit columns 0..3");
  extern __shared__ __align__(128) unsigned char sm[];

  const int K = KSPEC ? KSPEC : a.K;  // hidden size
  const int NW = K / 256, KG = KSPEC ? KGS : K / G, RB = K * BITS / 8;
  const int mt = MT1 ? 1 : a.mt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int rp = MT1 ? 1 : a.red_pitch, nb = a.nb;
  uint64_t* full_sb = reinterpret_cast<uint64_t*>(sm + a.off_bars);  // [kSBlocks] S/ZS landed
  uint64_t* red_empty = full_sb + kSBlocks;                            // [nb] partials consumed
  int* blk_cnt = reinterpret_cast<int*>(red_empty + kMaxRedBufs);      // [nb] warps done
  int* sz_issued = blk_cnt + kMaxRedBufs;                              // [kSBlocks] latest block
  int* job_done = sz_issued + kSBlocks;      // [nb] epilogue jobs finished per partial buffer
  int* job_pub = job_done + kMaxRedBufs;     // [nb] warp that published the buffer's jobs
  int* jobs_ready = job_pub + kMaxRedBufs;   // jobs [0, jobs_ready) may run
  int* jobs_claimed = jobs_ready + 1;        // jobs [0, jobs_claimed) taken by some warp
  volatile int* abort_flag = jobs_claimed + 1;
  float* xs_part = reinterpret_cast<float*>(sm + a.off_xs);  // [NW][8][NQ] strip group sums
  float* xs_full = xs_part + NW * 8 * NQ;                    // [mt][KG] group sums XS
  uint2* zb = reinterpret_cast<uint2*>(sm + a.off_zb);  // [KG/8][3][mt][4] B fragments of Z
  unsigned char* sz = sm + a.off_sz;                      // [kSBlocks][S|ZS][64][KG] bf16
  float* red = reinterpret_cast<float*>(sm + a.off_red);  // [nb][NW + 1][64][rp]
  const int sz_half = kBlockRows * KG * 2;                // bytes of a stage's S (or ZS) rows
  const int red_wstride = kBlockRows * rp;

  const int my_blocks = (a.nblk - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                        static_cast<int>(gridDim.x);
  auto block_row0 = [&](int lb) {
    return (static_cast<int>(blockIdx.x) + lb * static_cast<int>(gridDim.x)) * kBlockRows;
  };

  // S and ZS rows of local block lb into stage lb % kSBlocks (rows past N are not copied; the
  // epilogue ignores those rows). One thread.
  auto issue_sz = [&](int lb) {
    const int st = lb & (a.nsb - 1);
    const int row0 = block_row0(lb);
    sz_issued[st] = lb;
    int rows = a.N - row0;
    rows = rows > kBlockRows ? kBlockRows : rows;
    const uint32_t bytes = static_cast<uint32_t>(rows * KG * 2);  // multiple of 16: KG % 8 == 0
    mbar_arrive_expect_tx(&full_sb[st], 2u * bytes);
    unsigned char* dst = sz + st * 2 * sz_half;
    bulk_g2s(dst, a.S + static_cast<int64_t>(row0) * KG, bytes, &full_sb[st]);
    bulk_g2s(dst + sz_half, a.ZS + static_cast<int64_t>(row0) * KG, bytes, &full_sb[st]);
  };

  if (threadIdx.x == 0) {
    for (int q = 0; q < kSBlocks; ++q) mbar_init(&full_sb[q], 1u);
    for (int q = 0; q < kMaxRedBufs; ++q) {
      mbar_init(&red_empty[q], 1u);
      blk_cnt[q] = 0;
    }
    for (int q = 0; q < kMaxRedBufs; ++q) job_done[q] = job_pub[q] = 0;
    *jobs_ready = 0;
    *jobs_claimed = 0;
    *abort_flag = 0;
    mbar_fence_init();
    // the first S/ZS stages into L2 only (see the weight prefetch below); copied after the wait
    for (int lb = 0; lb < a.nsb && lb < my_blocks; ++lb) {
      const int row0 = block_row0(lb);
      const int rows = a.N - row0 > kBlockRows ? kBlockRows : a.N - row0;
      prefetch_l2_bulk(a.S + static_cast<int64_t>(row0) * KG, static_cast<uint32_t>(rows * KG * 2));
      prefetch_l2_bulk(a.ZS + static_cast<int64_t>(row0) * KG, static_cast<uint32_t>(rows * KG * 2));
    }
  }

  // ---- weight streaming of tile tau = 4 lb + t into ring stage tau % NSW, by warp `warp` alone:
  // chunk e = lane + 32 j is row e / (SB/16), 16-byte column e % (SB/16) of the warp's strip;
  // int4 rows are XOR-swizzled by (row & 1) so the two rows one quarter-warp reads use disjoint
  // banks; rows past N are zero-filled.
  const int strip_byte = warp * SB;
  constexpr int CPR = SB / 16;   // 16-byte chunks per strip row
  constexpr int RPJ = 32 / CPR;  // rows between a lane's successive chunks
  const int r0l = lane / CPR, col0 = lane % CPR;
  // the XOR swizzle depends on row parity only, and RPJ is even: the same for all of a lane's chunks
  const int pcol0 = BITS == 4 ? (col0 ^ ((r0l & 1) << 2)) : col0;
  const uint32_t dst_lane =
      smem_addr(sm + a.off_ring + warp * (NSW * WSTAGE)) + r0l * SB + 16 * pcol0;
  const int src_lane = strip_byte + 16 * col0;
  // Weight prefetch. blk_src(lbk): this lane's source pointer for local block lbk (row r0l of
  // the block), whether the block is one of this CTA's and whether it lies below N; computed
  // once per block, so a tile's copies use compile-time offsets from it. Past this CTA's blocks
  // the copies read nothing (zero-fill); in the block that crosses N, rows past N re-read row
  // N - 1 (their values are ignored).
  struct BlkSrc {
    const uint8_t* p;
    int row0;
    bool live, full;
  };
  auto blk_src = [&](int lbk) {
    BlkSrc b;
    b.row0 = block_row0(lbk);
    b.live = lbk < my_blocks;
    b.full = b.row0 + kBlockRows <= a.N;
    b.p = a.packed + static_cast<int64_t>(b.row0 + r0l) * RB + src_lane;
    return b;
  };
  // ring stage of tile tk of local block lbk: (4 lbk + tk) mod NSW
  auto ring_stage = [&](int lbk, int tk) { return (((4 * lbk) & (NSW - 1)) + tk) & (NSW - 1); };
  auto load_tile = [&](const BlkSrc& b, int lbk, int tk) {
    const uint32_t dst = dst_lane + ring_stage(lbk, tk) * WSTAGE;
    if (b.live && b.full) {
#pragma unroll
      for (int j = 0; j < CH; ++j)
        cp_async16(dst + j * RPJ * SB, b.p + static_cast<int64_t>(tk * kTileRows + j * RPJ) * RB,
                   true);
    } else {
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int rj = min(b.row0 + tk * kTileRows + r0l + j * RPJ, a.N - 1);
        cp_async16(dst + j * RPJ * SB,
                   b.live ? a.packed + static_cast<int64_t>(rj) * RB + src_lane : a.packed, b.live);
      }
    }
    cp_async_commit();  // one group per tile slot, possibly empty, keeps the counting uniform
  };
  // ---- weight prefetch: the first NSW - 1 tiles of this warp's strip (and, above, the S/ZS
  // stages) are fetched into L2 while the preceding kernel may still run. Only L2: the
  // preceding kernel's writes are guaranteed visible after griddepcontrol.wait alone, and it
  // may be the one that wrote the weights (the quantiser, or a caller's kernel); L2 is coherent,
  // so warming it early is safe, and the copies into shared memory come after the wait.
  {
    const BlkSrc b0 = blk_src(0), b1 = blk_src(1);
#pragma unroll
    for (int t = 0; t < NSW - 1; ++t) {
      const BlkSrc& b = t / kTilesPerBlock ? b1 : b0;
      const int tk = t % kTilesPerBlock;
      if (!b.live) continue;
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int rj = min(b.row0 + tk * kTileRows + r0l + j * RPJ, a.N - 1);
        prefetch_l2(a.packed + static_cast<int64_t>(rj) * RB + src_lane);
      }
    }
  }
  // Launched as a programmatic dependent: everything below (the weights into shared memory, x,
  // the outputs) waits for the preceding kernel's completion and the visibility of its writes
  // (a no-op after an ordinary launch).
  grid_dependency_wait();
  if (threadIdx.x == 0)
    for (int lb = 0; lb < a.nsb && lb < my_blocks; ++lb) issue_sz(lb);
  {
    const BlkSrc b0 = blk_src(0), b1 = blk_src(1);
#pragma unroll
    for (int t = 0; t < NSW - 1; ++t)
      load_tile(t / kTilesPerBlock ? b1 : b0, t / kTilesPerBlock, t % kTilesPerBlock);
  }

  // ---- this warp's view of x: the strip's values for the MMA's B operand. Lanes of column g
  // hold hidden row g (zeros for g >= mt); with one hidden row every lane holds it.
  const int xrow = MT1 ? 0 : (g < mt ? g : 0);
  const bool xval = MT1 || g < mt;
  const uint16_t* xg = a.x + static_cast<int64_t>(a.m0 + xrow) * K;
  uint2 xv[U][4][P];
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < P; ++p)
        xv[u][i][p] = xval ? *reinterpret_cast<const uint2*>(
                                 xg + p * (K / P) + strip_byte + 64 * u + 16 * c + 4 * i)
                           : make_uint2(0u, 0u);

  // S column of scale group q = (fold segment f, plane p) of this strip: p*(RB/G) + (strip+64f)/G
  auto s_col = [&](int q) {
    return (q % P) * (RB / G) + (strip_byte + 64 * (q / P)) / G;
  };
  auto pow2 = [](int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); };

  // B operand: x of the lane's hidden row for strip bytes 64u + 16c + 4i + {0, 2} (register 0)
  // and {1, 3} (register 1), plane p, as f16 x * s / 2^plane_shift(p). Each warp scales by its
  // own power of two s = 2^(15 - E), max |x| = f * 2^E (f in [0.5, 1)) over its strip of the
  // row, and converts its partials to logit units before storing them. With one hidden row,
  // scale group q has MMA column q: the lanes of column g hold only the values of their own group
  // q = g (lanes g >= NQ hold group 0's, their columns are never read), and every MMA takes the
  // lane's own values: column q of the accumulator of group q is then exact. Also the sums of x
  // over the strip's part of each scale group q.
  constexpr int BU = MT1 ? (SPLIT ? 1 : U) : U;  // B registers: [BU][4][BP][2]
  constexpr int BP = MT1 ? 1 : P;
  uint32_t bfr[BU][4][BP][2];
  const int q_own = MT1 && g < NQ ? g : 0;  // MT1: this lane's scale group
  const int u_own = SPLIT ? q_own / P : 0, p_own = q_own % P;
  int ew;  // E of this warp's strip of the lane's hidden row
  float xsg[NQ];
  {
    uint32_t mx = 0;  // max |x| as bf16 magnitude bits (monotone in the value)
#pragma unroll
    for (int q = 0; q < NQ; ++q) xsg[q] = 0.0f;
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const uint2 v = xv[u][i][p];
          mx = max(mx, max(max(v.x & 0x7fffu, (v.x >> 16) & 0x7fffu),
                           max(v.y & 0x7fffu, (v.y >> 16) & 0x7fffu)));
          xsg[(SPLIT ? u : 0) * P + p] += (bf16_bits_to_float(v.x & 0xffffu) + bf16_bits_to_float(v.x >> 16)) +
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
    for (int u = 0; u < BU; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) bfr[u][i][0][e] = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const float sx = pow2(15 - ew - plane_shift<BITS>(p));  // max |x * s| < 2^15
          const uint2 v = xv[u][i][p];
          const uint32_t h[4] = {v.x & 0xffffu, v.x >> 16, v.y & 0xffffu, v.y >> 16};
          uint32_t hs[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            hs[e] = __half_as_ushort(__float2half_rn(bf16_bits_to_float(h[e]) * sx));
          const uint32_t r0 = hs[0] | (hs[2] << 16);  // (x[k0], x[k0+2]): even bytes of the word
          const uint32_t r1 = hs[1] | (hs[3] << 16);  // (x[k0+1], x[k0+3]): odd bytes
          if (MT1) {
            if (p == p_own && (!SPLIT || u == u_own)) {
              bfr[SPLIT ? 0 : u][i][0][0] = r0;
              bfr[SPLIT ? 0 : u][i][0][1] = r1;
            }
          } else {
            bfr[u][i][MT1 ? 0 : p][0] = r0;
            bfr[u][i][MT1 ? 0 : p][1] = r1;
          }
        }
  }
  // Group sums XS[m][col] of the whole row (for the zero-point MMA): each warp publishes its
  // strip's part, then the parts of each group are added in warp order (deterministic).
  if (c == 0 && g < mt) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) xs_part[(warp * 8 + g) * NQ + q] = xsg[q];
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
      for (int w = r0 / SB; w <= (r0 + G - 1) / SB; ++w) {
        const int f = SPLIT ? (r0 - w * SB) / 64 : 0;
        sum += xs_part[(w * 8 + m) * NQ + f * P + p];
      }
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

  // byte offset of this lane's S entry of scale group q in a stage: so_g + 2 * s_col(q)
  // (row g of tile t adds t * 16 rows; row g + 8 adds row8)
  const int so_g = g * KG * 2;
  const int row8 = 8 * KG * 2;
  const unsigned char* ring = sm + a.off_ring + warp * (NSW * WSTAGE);
  float* rw_base = red + warp * red_wstride + g * rp + (MT1 ? 0 : 2 * c);

  // ---- zero-point part of a block, in logit units, into partial slot `zs` ([64][rp]): per
  // 16-row tile, sum over groups of (S - ZS) * XS as A = [S | ZS] (bf16, as stored) times
  // B = [XS ; -XS] in three bf16 parts; D layout (rows g, g + 8 x hidden rows 2c, 2c + 1).
  auto zero_point_block = [&](const unsigned char* stage, float* zs) {
    const uint2* zl = zb + (g < mt ? g : 0) * 4 + c;
    const bool zlive = g < mt;
#pragma unroll 1
    for (int t = 0; t < kTilesPerBlock; ++t) {
      float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
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
          mma_bf16_16816_acc(z, av[0], av[1], av[2], av[3], b.x, b.y);
        }
      }
      float* zw = zs + (t * kTileRows + g) * rp + (MT1 ? 0 : 2 * c);
      if (MT1) {
        if (c == 0) {
          zw[0] = z[0];
          zw[8] = z[2];
        }
      } else {
        if (2 * c < mt) {
          zw[0] = z[0];
          zw[8 * rp] = z[2];
        }
        if (2 * c + 1 < mt) {
          zw[1] = z[1];
          zw[8 * rp + 1] = z[3];
        }
      }
    }
  };

  // ---- epilogue job: top-KCAND of hidden row m of local block lb, partials in buf (the NW
  // warps' and the zero-point slot)
  auto epilogue = [&](int lb, int buf, int m) {
    const int b = static_cast<int>(blockIdx.x) + lb * static_cast<int>(gridDim.x);
    const int n0 = b * kBlockRows + lane;
    const float* rbuf = red + buf * (NW + 1) * red_wstride;
    {
      float v[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // fixed summation order (deterministic): four interleaved chains, then pairwise
        const float* rb = rbuf + (lane + 32 * h) * rp + m;
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
        int w = 0;
        for (; w + 4 <= NW + 1; w += 4) {
          s0 += rb[w * red_wstride];
          s1 += rb[(w + 1) * red_wstride];
          s2 += rb[(w + 2) * red_wstride];
          s3 += rb[(w + 3) * red_wstride];
        }
        for (; w < NW + 1; ++w) s0 += rb[w * red_wstride];
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
  };

  // ---- epilogue jobs: job j = lb * mt + m is hidden row m of local block lb; it may run once
  // jobs_ready > j (block lb complete). Every decision is lane 0's, broadcast, so that all lanes
  // take the same path (the epilogue holds warp-wide reductions).
  // own = false: leave jobs this warp published itself (it finished the block last: it is the
  // slowest warp) to the others.
  auto try_job = [&](bool own) -> bool {
    int j = -1;
    if (lane == 0) {
      const int cl = *reinterpret_cast<volatile int*>(jobs_claimed);
      if (cl < *reinterpret_cast<volatile int*>(jobs_ready) &&
          (own || *reinterpret_cast<volatile int*>(&job_pub[(MT1 ? cl : cl / mt) & (nb - 1)]) != warp) &&
          atomicCAS(jobs_claimed, cl, cl + 1) == cl)
        j = cl;
    }
    j = __shfl_sync(0xffffffffu, j, 0);
    if (j < 0) return false;
    const int jb = MT1 ? j : j / mt, m = MT1 ? 0 : j - jb * mt, jbuf = jb & (nb - 1);
    __syncwarp();
    __threadfence_block();  // the block's partials, published before jobs_ready, are visible
    epilogue(jb, jbuf, m);
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (MT1 || atomicAdd(&job_done[jbuf], 1) == mt - 1) {  // the block's last job
        if (!MT1) job_done[jbuf] = 0;
        mbar_arrive(&red_empty[jbuf]);
      }
    }
    return true;
  };
  // Bounded wait for phase `parity` of `bar`: runs an epilogue job if one is ready, else lane 0
  // sleeps in the mbarrier (woken when the phase completes, or after a few microseconds to look
  // for jobs again). False after a timeout (the launch is marked failed) or another warp's.
  auto wait_taking_jobs = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint64_t t0 = global_timer_ns();
    while (true) {
      int st = 0;
      if (lane == 0) st = mbar_test_wait(bar, parity) ? 1 : (*abort_flag ? -1 : 0);
      st = __shfl_sync(0xffffffffu, st, 0);
      if (st > 0) {
        mbar_test_wait(bar, parity);  // every lane acquires (the phase stays complete)
        return true;
      }
      if (st < 0) return false;
      if (try_job(true)) continue;
      if (lane == 0) mbar_try_wait_ns(bar, parity, 4000u);
      __syncwarp();
      if (lane == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        set_status(a.status, DH_DEV_WAIT_TIMEOUT);
      }
    }
  };

  // factor kappa / s that turns this lane's partials into logits: hidden rows 2c, 2c + 1 (MT1:
  // the one hidden row, in ysc[0])
  float ysc[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int hr = MT1 ? 0 : 2 * c + j, src = (hr < 8 ? hr : 0) * 4;
    const int e = __shfl_sync(0xffffffffu, ew, src);
    ysc[j] = hr < mt ? pow2(e + 9 - kLogL) : 0.0f;
  }
  // MT1: the two scale groups (columns 2c, 2c + 1) this lane folds; lanes past NQ/2 hold zero
  // columns and fold a valid group's scale into them (no effect).
  const int qa = MT1 ? (2 * c < NQ ? 2 * c : 0) : 0;
  const int soa = so_g + 2 * s_col(qa), sob = so_g + 2 * s_col(qa + 1 < NQ ? qa + 1 : qa);
  // The last of the block's NW + 1 arrivals (every warp, plus the zero-point pass) refills the
  // block's S/ZS stage and publishes its epilogue jobs. Lane 0.
  auto finish_block = [&](int lb, int buf) {
    blk_cnt[buf] = 0;
    __threadfence_block();
    if (lb + a.nsb < my_blocks) {
      fence_proxy_async_smem();  // stage reads happen before the copy's writes
      issue_sz(lb + a.nsb);
    }
    job_pub[buf] = warp;
    __threadfence_block();
    atomicMax(jobs_ready, (lb + 1) * mt);
  };

  for (int lb = 0; lb < my_blocks; ++lb) {
    const int buf = lb & (nb - 1), sst = lb & (a.nsb - 1);
    {
      bool ok = wait_taking_jobs(&full_sb[sst], static_cast<uint32_t>(lb >> a.nsb_log) & 1u);
      if (ok && lb >= nb)
        ok = wait_taking_jobs(&red_empty[buf], static_cast<uint32_t>(lb / nb - 1) & 1u);
      if (!ok) break;
      try_job(false);  // an epilogue another warp published, if one is ready
    }
    const unsigned char* stage = sz + sst * 2 * sz_half;
    float* rwb = rw_base + buf * (NW + 1) * red_wstride;
    // the prefetches of this block's tiles target blocks lb + kA and lb + kA + 1
    constexpr int kA = (NSW - 1) / kTilesPerBlock;
    const BlkSrc bA = blk_src(lb + kA), bB = blk_src(lb + kA + 1);
#pragma unroll
    for (int t = 0; t < kTilesPerBlock; ++t) {
      {
        const int pt = t + NSW - 1, pb = pt / kTilesPerBlock - kA, ptk = pt % kTilesPerBlock;
        load_tile(pb ? bB : bA, lb + kA + pb, ptk);
      }
      cp_async_wait<NSW - 1>();  // tile (lb, t) has landed (for this lane's copies)
      __syncwarp();              // ... and for every lane's
      const unsigned char* cs = ring + ring_stage(lb, t) * WSTAGE;
      const unsigned char* szs = stage + t * (kTileRows * KG * 2);
      float acc[4];
      if (MT1) {
        // one accumulator per scale group q (four independent chains); column q of dq[q] is
        // group q's dot, the other columns are ignored
        float dq[NQ][4];
#pragma unroll
        for (int q = 0; q < NQ; ++q) dq[q][0] = dq[q][1] = dq[q][2] = dq[q][3] = 0.0f;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int pc = BITS == 4 ? ((4 * u + c) ^ ((g & 1) << 2)) : c;  // swizzled column
          const uint4 wa = *reinterpret_cast<const uint4*>(cs + g * SB + 16 * pc);
          const uint4 wb = *reinterpret_cast<const uint4*>(cs + (g + 8) * SB + 16 * pc);
          const uint32_t ta[4] = {wa.x, wa.y, wa.z, wa.w}, tb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t tao = ta[i] >> 8, tbo = tb[i] >> 8;
#pragma unroll
            for (int p = 0; p < P; ++p)
              mma_f16_16816_acc(dq[(SPLIT ? u * P : 0) + p], dq16<BITS>(ta[i], p),
                                dq16<BITS>(tb[i], p), dq16<BITS>(tao, p), dq16<BITS>(tbo, p),
                                bfr[SPLIT ? 0 : u][i][0][0], bfr[SPLIT ? 0 : u][i][0][1]);
          }
        }
        // lane c holds columns 2c, 2c + 1: group 2c in dq[2c][0, 2], group 2c + 1 in
        // dq[2c + 1][1, 3] (rows g, g + 8)
        float da0, da2, db1, db3;
        if (NQ > 2) {
          const bool hi = c & 1;  // lanes c = 2, 3 only pair with each other below
          da0 = hi ? dq[NQ > 2 ? 2 : 0][0] : dq[0][0];
          da2 = hi ? dq[NQ > 2 ? 2 : 0][2] : dq[0][2];
          db1 = hi ? dq[NQ > 3 ? 3 : 1][1] : dq[1][1];
          db3 = hi ? dq[NQ > 3 ? 3 : 1][3] : dq[1][3];
        } else {
          da0 = dq[0][0];
          da2 = dq[0][2];
          db1 = dq[NQ > 1 ? 1 : 0][1];
          db3 = dq[NQ > 1 ? 1 : 0][3];
        }
        const float sa = __uint_as_float(lds_u16(szs + soa) * a.u16_mul);
        const float sb = __uint_as_float(lds_u16(szs + sob) * a.u16_mul);
        const float sa8 = __uint_as_float(lds_u16(szs + soa + row8) * a.u16_mul);
        const float sb8 = __uint_as_float(lds_u16(szs + sob + row8) * a.u16_mul);
        float r0 = fmaf(sb, db1, sa * da0);
        float r8 = fmaf(sb8, db3, sa8 * da2);
        if (NQ > 2) {  // groups 2, 3 sit in lane c = 1
          r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
          r8 += __shfl_xor_sync(0xffffffffu, r8, 1);
        }
        acc[0] = r0;
        acc[2] = r8;
        acc[1] = acc[3] = 0.0f;
      } else {
        acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
        float d[P][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int pc = BITS == 4 ? ((4 * u + c) ^ ((g & 1) << 2)) : c;  // swizzled column
          const uint4 wa = *reinterpret_cast<const uint4*>(cs + g * SB + 16 * pc);
          const uint4 wb = *reinterpret_cast<const uint4*>(cs + (g + 8) * SB + 16 * pc);
          const uint32_t ta[4] = {wa.x, wa.y, wa.z, wa.w}, tb[4] = {wb.x, wb.y, wb.z, wb.w};
          uint32_t tao[4], tbo[4];  // odd bytes moved down: t >> 8
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            tao[i] = ta[i] >> 8;
            tbo[i] = tb[i] >> 8;
          }
          const int f = SPLIT ? u : 0;
          const bool seg_first = SPLIT || u == 0, seg_last = SPLIT || u == U - 1;
          // plane by plane: the plane's accumulator is folded as soon as its segment is complete
#pragma unroll
          for (int p = 0; p < P; ++p) {
            if (seg_first) {
#pragma unroll
              for (int e = 0; e < 4; ++e) d[p][e] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma_f16_16816_acc(d[p], dq16<BITS>(ta[i], p), dq16<BITS>(tb[i], p),
                                dq16<BITS>(tao[i], p), dq16<BITS>(tbo[i], p),
                                bfr[u][i][MT1 ? 0 : p][0], bfr[u][i][MT1 ? 0 : p][1]);
            if (seg_last) {
              const unsigned char* sq = szs + so_g + 2 * s_col(f * P + p);
              const float sg = __uint_as_float(lds_u16(sq) * a.u16_mul);
              const float sg8 = __uint_as_float(lds_u16(sq + row8) * a.u16_mul);
              acc[0] = fmaf(sg, d[p][0], acc[0]);
              acc[1] = fmaf(sg, d[p][1], acc[1]);
              acc[2] = fmaf(sg8, d[p][2], acc[2]);
              acc[3] = fmaf(sg8, d[p][3], acc[3]);
            }
          }
        }
      }
      // partials in logit units, D layout: acc[0..1] = row g, hidden rows 2c, 2c+1; acc[2..3] =
      // row g + 8 (MT1: acc[0], acc[2] in lane c = 0)
      float* rw = rwb + t * kTileRows * rp;
      if (MT1) {
        if (c == 0) {
          rw[0] = acc[0] * ysc[0];
          rw[8] = acc[2] * ysc[0];
        }
      } else {
        if (2 * c < mt) {
          rw[0] = acc[0] * ysc[0];
          rw[8 * rp] = acc[2] * ysc[0];
        }
        if (2 * c + 1 < mt) {
          rw[1] = acc[1] * ysc[1];
          rw[8 * rp + 1] = acc[3] * ysc[1];
        }
      }
    }
    // end of block lb for this warp: the first warp here also computes the block's zero-point
    // slot (the S/ZS stage stays until every arrival, that pass's included, is in)
    __syncwarp();  // every lane's partial stores and stage reads are done
    int first = 0;
    if (lane == 0) {
      __threadfence_block();
      const int old = atomicAdd(&blk_cnt[buf], 1);
      first = old == 0;
      if (old == NW) finish_block(lb, buf);
    }
    if (__shfl_sync(0xffffffffu, first, 0)) {
      zero_point_block(stage, red + buf * (NW + 1) * red_wstride + NW * red_wstride);
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(&blk_cnt[buf], 1) == NW) finish_block(lb, buf);
      }
    }
  }
  // drain. One job per block: take the jobs that are ready, then leave (every block's jobs are
  // published by a warp before it drains, so the warp that publishes the last block takes
  // whatever is left).
  if (MT1) {
    while (try_job(true)) {
    }
  } else {
    // several jobs per block: wait (sleeping) for the rest, so the last blocks' jobs run in
    // parallel on the warps that are done rather than one after another on the last publisher
    const uint64_t t0 = global_timer_ns();
    while (true) {
      int st = 0;
      if (lane == 0)
        st = *reinterpret_cast<volatile int*>(jobs_claimed) >= my_blocks * mt || *abort_flag;
      if (__shfl_sync(0xffffffffu, st, 0)) break;
      if (try_job(true)) continue;
      __nanosleep(1000);
      if (lane == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        set_status(a.status, DH_DEV_WAIT_TIMEOUT);
      }
    }
  }
  cp_async_wait<0>();
  // After an abort, S/ZS copies may still be in flight: they must land before the CTA's shared
  // memory goes away. (Normally every issued stage has been waited for already.)
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    for (int q = 0; q < a.nsb && q < my_blocks; ++q)
      mbar_wait_bounded(&full_sb[q], static_cast<uint32_t>(sz_issued[q] >> a.nsb_log) & 1u);
  }
}


// Launches one pass (hidden rows m0 .. m0 + mt - 1) of the kernel for a given plan: the hidden
// size is compiled in for K = 5120, the single-row case for mt = 1.
template <int BITS, int G>
cudaError_t launch_coarse_variant(const CoarseArgs& a, int nsw, int grid, cudaStream_t s) {
  auto go = [&](auto kernel) -> cudaError_t {
    constexpr int SB = BITS == 2 ? 64 : 128;
    const int smem = a.off_ring + a.NW * nsw * kTileRows * SB;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the CTAs may start (and prefetch weights) while the kernel
    // before them in the stream finishes, once it lets its dependents start
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(a.NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  };
  auto by_nsw = [&](auto kspec, auto mt1) -> cudaError_t {
    constexpr int KS = decltype(kspec)::value;
    constexpr bool M1 = decltype(mt1)::value;
    switch (nsw) {
      case 8: return go(coarse_topk_kernel<BITS, G, KS, 8, M1>);
      case 4: return go(coarse_topk_kernel<BITS, G, KS, 4, M1>);
      default: return go(coarse_topk_kernel<BITS, G, KS, 2, M1>);
    }
  };
  using K0 = std::integral_constant<int, 0>;
  using K5120 = std::integral_constant<int, 5120>;
  using T = std::true_type;
  using F = std::false_type;
  if (a.K == 5120) return a.mt == 1 ? by_nsw(K5120{}, T{}) : by_nsw(K5120{}, F{});
  return a.mt == 1 ? by_nsw(K0{}, T{}) : by_nsw(K0{}, F{});
}

}  // namespace dh
