// Coarse pass + block top-KCAND of the low-bit draft head (page "radiance_drafthead.py":
// module docstring, _draft_head_int2 and _emit), for sm_103a.
//
// Work decomposition (GB300-first, not the page's one-program-per-block grid):
//  * Persistent grid, one CTA per SM. A CTA walks 64-row candidate blocks b = blockIdx.x,
//    blockIdx.x + gridDim.x, ...; each block is four 16-row tiles.
//  * NW = K/256 warps. Warp w owns the same 256 k-values of every vocab row (its "strip":
//    bytes [64w, 64w+64) of each int2 row, [128w, 128w+128) of each int4 row). So:
//      - its share of the hidden states never changes: the permuted x fragments of the MMA's B
//        operand live in registers for the whole launch;
//      - it streams only its own strip of each tile (16 rows x 64 B) through a private ring of
//        shared-memory stages with 16-byte cp.async copies, NSW-1 tiles ahead: no warp ever
//        waits on another warp for weights.
//  * Per tile the warp dequantises its strip with the page's bit patterns straight into MMA A
//    fragments (0x3F80 | ((b << (5-2q)) & 0x60) = 1 + v/4 for int2, 0x3F80 | (nibble << 3) =
//    1 + v/16 for int4; weights on the MMA's 16-row side, hidden rows on its 8-column side) and
//    issues mma.sync m16n8k16 (bf16 in, fp32 accumulate, in place). The MMA's k order is
//    permuted so that bytes j and j+2 of a 32-bit word share one bf16x2 register; x is permuted
//    the same way.
//  * The per-group scale is applied to the accumulator, never to the weight tile:
//    acc += S[n,g] * P_g for each (plane, group) of the strip; the warp streams the S entries it
//    needs into the same ring stage as the tile's weights.
//  * Block epilogue by shared job tickets: every warp writes its partial sums of the block into a
//    double buffer and moves on; the last warp to finish the block publishes the block's jobs
//    (one per hidden row); any warp at a tile boundary takes the next published job: it sums the
//    NW partials in warp order (deterministic), subtracts the zero-point term
//    sum_g ZS[n,g] * XS[m,g] in fp32, selects with warp reductions (max key, then lowest row on
//    ties) and writes the candidates. A warp that must wait for a buffer takes jobs meanwhile.
// Hidden rows are processed eight at a time (one MMA column tile); M > 8 runs ceil(M/8) passes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dh_device.cuh"
#include "dh_launch.h"

namespace dh {

constexpr int kCoarseMaxWarps = 20;  // K <= 5120
constexpr int kCoarseMaxThreads = kCoarseMaxWarps * 32;

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
  // Power-of-two multipliers of the dequant, one per plane (see dq below). They arrive as kernel
  // parameters so the shift-and-OR stays an integer multiply-add on the FMA pipe.
  uint32_t dq_mul[4];
  // shared-memory layout (bytes)
  int nbuf, red_pitch, ring_warp_bytes;
  int off_ring, off_red, off_xs, off_bars;
};

// Bit-pattern dequant of one plane of a 32-bit word t (bytes b0..b3) into a bf16x2 register:
// the plane's code v of byte 0 goes to the low half and of byte 2 to the high half, as the bf16
// value 1 + v/4 (int2, pattern 0x3F80 | v << 5) or 1 + v/16 (int4, 0x3F80 | v << 3). Bytes 1 and 3
// use the same function on t >> 8. The code bits are masked in place (LOP3, ALU pipe) and moved
// to their mantissa slot with the 0x3F80 exponent added in one integer multiply-add (IMAD or
// IMAD.HI, FMA pipe): since the masked bits and 0x3F803F80 do not overlap, + is |. For int2 this
// is exactly the page's 0x3F80 | ((b << (5-2q)) & 0x60) (q < 3) and 0x3F80 | ((b >> 1) & 0x60)
// (q = 3), evaluated on two bytes at once.
__device__ __forceinline__ uint32_t mad_lo_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t mad_hi_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int BITS>
__device__ __forceinline__ uint32_t dq(uint32_t t, int p, const uint32_t (&mul)[4]) {
  constexpr uint32_t kOne = 0x3F803F80u;  // bf16x2 (1.0, 1.0)
  if (BITS == 2) {
    // plane p at bits 2p, 2p+1 of each byte -> bits 5, 6: x 2^(5-2p) for p < 3, x 2^-1 for p = 3
    const uint32_t m = t & (0x00030003u << (2 * p));
    return p < 3 ? mad_lo_u32(m, mul[p], kOne) : mad_hi_u32(m, mul[3], kOne);
  } else {
    // nibble p at bits 4p .. 4p+3 -> bits 3 .. 6: x 2^3 for p = 0, x 2^-1 for p = 1
    const uint32_t m = t & (0x000F000Fu << (4 * p));
    return p == 0 ? mad_lo_u32(m, mul[0], kOne) : mad_hi_u32(m, mul[1], kOne);
  }
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem_dst)),
               "l"(gsrc), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(smem_dst)),
               "l"(gsrc), "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// SPLIT: the strip spans more than one quantisation group per plane (int4 with G = 64), so the
// accumulator is folded once per 64-byte sub-chunk instead of once per strip.
// NSW: stages of each warp's private ring.
template <int BITS, bool SPLIT, int NSW>
__global__ void __launch_bounds__(kCoarseMaxThreads, 1) coarse_topk_kernel(const CoarseArgs a) {
  constexpr int P = 8 / BITS;                 // codes per byte (planes)
  constexpr int SB = 256 / P;                 // strip bytes per row: 256 k-values
  constexpr int U = SB / 64;                  // 64-byte sub-chunks per strip
  constexpr int FS = SPLIT ? U : 1;           // fold segments per strip
  constexpr int NQ = FS * P;                  // scale groups per strip
  constexpr int WSTAGE = kTileRows * SB;      // packed bytes of one warp's strip of a tile
  constexpr int STAGE = WSTAGE + NQ * kTileRows * 4;  // + the tile's scale words
  constexpr int CH = WSTAGE / 16 / 32;        // 16-byte weight copies per lane per tile
  constexpr int CS = NQ * kTileRows / 32;     // 4-byte scale copies per lane per tile
  static_assert((NSW & (NSW - 1)) == 0, "ring depth must be a power of two");
  extern __shared__ __align__(128) unsigned char sm[];

  const int NW = a.NW, KG = a.KG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int rp = a.red_pitch;
  uint64_t* red_empty = reinterpret_cast<uint64_t*>(sm + a.off_bars);  // [2] buffer released
  int* blk_arrived = reinterpret_cast<int*>(red_empty + 2);           // [2] warps done with block
  int* blk_jobs_done = blk_arrived + 2;                                // [2] jobs done per block
  int* jobs_ready = blk_jobs_done + 2;                                 // jobs published
  int* jobs_claimed = jobs_ready + 1;                                  // jobs taken
  volatile int* abort_flag = jobs_claimed + 1;
  float* xs_s = reinterpret_cast<float*>(sm + a.off_xs);              // [8][KG]
  float* red = reinterpret_cast<float*>(sm + a.off_red);              // [2][NW][64][rp]
  unsigned char* ring = sm + a.off_ring + warp * (NSW * STAGE);       // [NSW][STAGE]
  const int red_wstride = kBlockRows * rp;

  const int my_blocks = (a.nblk - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                        static_cast<int>(gridDim.x);
  const int my_tiles = my_blocks * kTilesPerBlock;
  const int strip_byte = warp * SB;
  // first vocab row of this CTA's tile tau
  auto tile_row0 = [&](int tau) {
    return (static_cast<int>(blockIdx.x) + (tau >> 2) * static_cast<int>(gridDim.x)) * kBlockRows +
           (tau & 3) * kTileRows;
  };
  // S column of scale group q = (fold segment f, plane p) of this strip: p*(RB/G) + (strip+64f)/G
  auto s_col = [&](int q) {
    return (q % P) * (a.RB / a.G) + (strip_byte + 64 * (q / P)) / a.G;
  };

  // ---- streaming of tile tau into ring stage tau % NSW, by this warp alone:
  //  * packed weights: chunk e = lane + 32 j is row e / (SB/16), 16-byte column e % (SB/16) of
  //    the warp's strip; int4 rows are XOR-swizzled by (row & 1) so the two rows one quarter-warp
  //    reads use disjoint banks;
  //  * scales: word e = lane + 32 j is the aligned bf16 pair holding S[row0 + e % 16][s_col(e / 16)];
  //  * rows past N are zero-filled.
  auto load_tile = [&](int tau) {
    if (tau < my_tiles) {
      const int row0 = tile_row0(tau);
      unsigned char* dst = ring + (tau & (NSW - 1)) * STAGE;
      const uint8_t* src = a.packed + static_cast<int64_t>(row0) * a.RB + strip_byte;
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int e = lane + 32 * j;
        const int r = e / (SB / 16), col = e % (SB / 16);
        const int pcol = BITS == 4 ? (col ^ ((r & 1) << 2)) : col;
        const bool ok = row0 + r < a.N;
        cp_async16(dst + r * SB + 16 * pcol, ok ? src + r * a.RB + 16 * col : a.packed, ok);
      }
#pragma unroll
      for (int j = 0; j < CS; ++j) {
        const int e = lane + 32 * j;
        const int r = e & (kTileRows - 1), q = e / kTileRows;
        const bool ok = row0 + r < a.N;
        const uint16_t* ssrc = a.S + static_cast<int64_t>(row0 + r) * KG + (s_col(q) & ~1);
        cp_async4(dst + WSTAGE + 4 * e, ok ? ssrc : a.S, ok);
      }
    }
    cp_async_commit();  // one group per tile slot, possibly empty, keeps the counting uniform
  };

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      mbar_init(&red_empty[q], 1u);
      blk_arrived[q] = 0;
      blk_jobs_done[q] = 0;
    }
    *jobs_ready = 0;
    *jobs_claimed = 0;
    *abort_flag = 0;
    mbar_fence_init();
  }
  // start streaming before the setup below
#pragma unroll
  for (int t = 0; t < NSW - 1; ++t) load_tile(t);

  // permuted x fragments of this warp's strip (B operand), kept in registers
  uint32_t bfr[U][4][P][2];
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < P; ++p) {
        uint32_t b0 = 0, b1 = 0;
        if (g < a.mt) {
          const int k0 = p * (a.K / P) + strip_byte + 64 * u + 16 * c + 4 * i;
          const uint2 v = *reinterpret_cast<const uint2*>(
              a.x + static_cast<int64_t>(a.m0 + g) * a.K + k0);
          b0 = __byte_perm(v.x, v.y, 0x5410);  // (x[k0], x[k0+2]): even bytes of the word
          b1 = __byte_perm(v.x, v.y, 0x7632);  // (x[k0+1], x[k0+3]): odd bytes
        }
        bfr[u][i][p][0] = b0;
        bfr[u][i][p][1] = b1;
      }

  // group sums of x in fp32, for the zero-point term
  for (int pr = warp; pr < a.mt * KG; pr += NW) {
    const int tok = pr / KG, gi = pr - tok * KG;
    const uint16_t* xr = a.x + static_cast<int64_t>(a.m0 + tok) * a.K + gi * a.G;
    float sum = 0.0f;
    for (int t = lane; t < a.G; t += 32) sum += bf16_bits_to_float(xr[t]);
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) xs_s[tok * KG + gi] = sum;
  }
  __syncthreads();

  // ---- epilogue job: top-KCAND of hidden row m of block b, partials in buffer buf ------------
  auto epilogue = [&](int b, int buf, int m) {
    const float* rb = red + buf * NW * red_wstride + m;
    const int n0 = b * kBlockRows + lane;
    float v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = lane + 32 * h;
      float s = 0.0f;
      for (int w = 0; w < NW; ++w) s += rb[w * red_wstride + row * rp];
      // zero-point term: - sum_g ZS[n, g] * XS[m, g], fp32, group order
      const int n = n0 + 32 * h;
      if (n < a.N) {
        const uint4* zr = reinterpret_cast<const uint4*>(a.ZS + static_cast<int64_t>(n) * KG);
        const float* xs = xs_s + m * KG;
        float z = 0.0f;
        for (int q = 0; q < KG / 8; ++q) {
          const uint4 zz = zr[q];
          const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            z = fmaf(__uint_as_float(zw[e] << 16), xs[8 * q + 2 * e], z);
            z = fmaf(__uint_as_float(zw[e] & 0xffff0000u), xs[8 * q + 2 * e + 1], z);
          }
        }
        s -= z;
      }
      v[h] = s;
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
  };

  // ---- shared job tickets: job c is hidden row c % mt of local block c / mt. The last warp to
  // finish a block publishes its mt jobs; any warp at a tile boundary takes the next published
  // job; the warp finishing a block's last job releases that block's partial buffer.
  const int total_jobs = my_blocks * a.mt;
  auto try_job = [&]() -> bool {
    int c = -1;
    if (lane == 0) {
      const int ready = *reinterpret_cast<volatile int*>(jobs_ready);
      int cl = *reinterpret_cast<volatile int*>(jobs_claimed);
      while (cl < ready) {
        const int prev = atomicCAS(jobs_claimed, cl, cl + 1);
        if (prev == cl) {
          c = cl;
          break;
        }
        cl = prev;
      }
      __threadfence_block();
    }
    c = __shfl_sync(0xffffffffu, c, 0);
    if (c < 0) return false;
    __threadfence_block();  // the partials published before the ticket are visible to every lane
    const int jbl = c / a.mt, m = c - jbl * a.mt;
    const int jbuf = jbl & 1;
    epilogue(static_cast<int>(blockIdx.x) + jbl * static_cast<int>(gridDim.x), jbuf, m);
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&blk_jobs_done[jbuf], 1) == a.mt - 1) {
        blk_jobs_done[jbuf] = 0;
        __threadfence_block();
        mbar_arrive(&red_empty[jbuf]);
      }
    }
    return true;
  };

  // ---- main loop over this CTA's tiles
  const int sh_lo = (s_col(0) & 1) * 16;  // half of the stored scale pair holding our column
  for (int tau = 0; tau < my_tiles; ++tau) {
    load_tile(tau + NSW - 1);              // into the stage the previous tile freed
    cp_async_wait<NSW - 1>();              // tile tau has landed (for this lane's copies)
    __syncwarp();                          // ... and for every lane's
    const int t = tau & 3, lb = tau >> 2, buf = lb & 1;

    if (t == 0 && lb >= 2) {
      // partial buffer reuse: block lb - 2 must have released it; take jobs while waiting
      // Every decision in this loop is lane 0's, broadcast: try_job holds warp-wide collectives,
      // so all lanes must take the same path even if they observe shared memory at different
      // moments.
      const uint32_t par = (static_cast<uint32_t>(lb >> 1) & 1u) ^ 1u;
      const uint64_t t0 = global_timer_ns();
      while (true) {
        const bool done = __shfl_sync(0xffffffffu,
                                      lane == 0 && (*abort_flag || mbar_test_wait(&red_empty[buf], par)),
                                      0);
        if (done) break;
        if (try_job()) continue;
        __nanosleep(64);
        if (lane == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
          *abort_flag = 1;
          set_status(a.status, DH_DEV_WAIT_TIMEOUT);
        }
      }
    }

    const unsigned char* cs = ring + (tau & (NSW - 1)) * STAGE;
    float d[FS][P][4];
#pragma unroll
    for (int f = 0; f < FS; ++f)
#pragma unroll
      for (int p = 0; p < P; ++p)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[f][p][e] = 0.0f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int pc = BITS == 4 ? ((4 * u + c) ^ ((g & 1) << 2)) : c;  // swizzled column
      const uint4 wa = *reinterpret_cast<const uint4*>(cs + g * SB + 16 * pc);
      const uint4 wb = *reinterpret_cast<const uint4*>(cs + (g + 8) * SB + 16 * pc);
      const uint32_t wav[4] = {wa.x, wa.y, wa.z, wa.w};
      const uint32_t wbv[4] = {wb.x, wb.y, wb.z, wb.w};
      const int f = SPLIT ? u : 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t wao = wav[i] >> 8, wbo = wbv[i] >> 8;  // odd bytes
#pragma unroll
        for (int p = 0; p < P; ++p)
          mma_bf16_16816_acc(d[f][p], dq<BITS>(wav[i], p, a.dq_mul),
                             dq<BITS>(wbv[i], p, a.dq_mul), dq<BITS>(wao, p, a.dq_mul),
                             dq<BITS>(wbo, p, a.dq_mul), bfr[u][i][p][0], bfr[u][i][p][1]);
      }
    }
    // scale on the accumulator: acc += S[n, g] * P_g (scale words of rows g and g + 8)
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(cs + WSTAGE);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int f = 0; f < FS; ++f)
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const int q = f * P + p;
        const int sh = (s_col(q) & 1) * 16;  // same parity for every q of a strip when SB >= G
        const float sg = __uint_as_float((sw[q * kTileRows + g] >> (FS == 1 ? sh_lo : sh)) << 16);
        const float sg8 =
            __uint_as_float((sw[q * kTileRows + g + 8] >> (FS == 1 ? sh_lo : sh)) << 16);
        acc[0] = fmaf(sg, d[f][p][0], acc[0]);
        acc[1] = fmaf(sg, d[f][p][1], acc[1]);
        acc[2] = fmaf(sg8, d[f][p][2], acc[2]);
        acc[3] = fmaf(sg8, d[f][p][3], acc[3]);
      }
    // partials, D layout: acc[0..1] = row g, hidden rows 2c, 2c+1; acc[2..3] = row g + 8
    float* rw = red + (buf * NW + warp) * red_wstride + (t * kTileRows + g) * rp + 2 * c;
    if (2 * c < a.mt) {
      rw[0] = acc[0];
      rw[8 * rp] = acc[2];
    }
    if (2 * c + 1 < a.mt) {
      rw[1] = acc[1];
      rw[8 * rp + 1] = acc[3];
    }
    __syncwarp();  // every lane is done with this stage and its partial stores are visible
    if (t == kTilesPerBlock - 1 && lane == 0) {
      __threadfence_block();
      if (atomicAdd(&blk_arrived[buf], 1) == NW - 1) {  // last warp: publish the block's jobs
        blk_arrived[buf] = 0;
        __threadfence_block();
        atomicAdd(jobs_ready, a.mt);
      }
    }
    try_job();
  }
  // drain: take jobs until every job of this CTA has been claimed and finished
  {
    const uint64_t t0 = global_timer_ns();
    while (true) {
      if (__shfl_sync(0xffffffffu, lane == 0 && *abort_flag != 0, 0)) break;  // uniform, as above
      if (try_job()) continue;
      if (__shfl_sync(0xffffffffu,
                      lane == 0 && *reinterpret_cast<volatile int*>(jobs_claimed) >= total_jobs, 0))
        break;
      __nanosleep(128);
      if (lane == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        set_status(a.status, DH_DEV_WAIT_TIMEOUT);
      }
    }
  }
  cp_async_wait<0>();
}

// Shared-memory plan for one launch; returns the ring depth (0 if nothing fits).
template <int BITS>
static int plan_coarse(CoarseArgs& a, int max_smem, int nsw_max) {
  constexpr int SB = BITS == 2 ? 64 : 128;
  a.RB = a.K * BITS / 8;
  a.KG = a.K / a.G;
  a.NW = a.K / 256;
  const int mt_max = a.M < 8 ? a.M : 8;
  a.red_pitch = mt_max | 1;  // odd: a warp reading one column over 32 rows hits 32 banks
  a.nbuf = 2;
  const int nq = (8 / BITS) * ((BITS == 4 && a.G < 128) ? 2 : 1);
  const int stage = kTileRows * SB + nq * kTileRows * 4;
  int off = 0;
  a.off_bars = off;
  off += 2 * 8 + 8 * 4 + 16;
  a.off_xs = off = (off + 15) / 16 * 16;
  off += 8 * a.KG * 4;
  a.off_red = off = (off + 15) / 16 * 16;
  off += 2 * a.NW * kBlockRows * a.red_pitch * 4;
  a.off_ring = off = (off + 127) / 128 * 128;
  for (int nsw = nsw_max; nsw >= 2; nsw /= 2) {
    a.ring_warp_bytes = nsw * stage;
    if (a.off_ring + a.NW * a.ring_warp_bytes <= max_smem) return nsw;
  }
  return 0;
}

template <int BITS, bool SPLIT, int NSW>
static cudaError_t launch_one(const CoarseArgs& a, int grid, cudaStream_t s) {
  const int smem = a.off_ring + a.NW * a.ring_warp_bytes;
  cudaError_t e = cudaFuncSetAttribute(coarse_topk_kernel<BITS, SPLIT, NSW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  coarse_topk_kernel<BITS, SPLIT, NSW><<<grid, a.NW * 32, smem, s>>>(a);
  return cudaGetLastError();
}

template <int BITS, bool SPLIT>
static cudaError_t launch_nsw(const CoarseArgs& a, int nsw, int grid, cudaStream_t s) {
  switch (nsw) {
    case 8: return launch_one<BITS, SPLIT, 8>(a, grid, s);
    case 4: return launch_one<BITS, SPLIT, 4>(a, grid, s);
    default: return launch_one<BITS, SPLIT, 2>(a, grid, s);
  }
}

// Returns cudaErrorInvalidValue if the shape does not fit the kernel's plan.
cudaError_t launch_coarse_topk(const CoarseCall& cc, int num_sms, int max_smem, cudaStream_t s) {
  CoarseArgs a{};
  a.x = static_cast<const uint16_t*>(cc.x);
  a.M = static_cast<int>(cc.M);
  a.K = static_cast<int>(cc.K);
  a.N = static_cast<int>(cc.N);
  a.G = cc.G;
  a.packed = cc.packed;
  a.S = static_cast<const uint16_t*>(cc.S);
  a.ZS = static_cast<const uint16_t*>(cc.ZS);
  a.kcand = cc.kcand;
  a.nblk = static_cast<int>((cc.N + kBlockRows - 1) / kBlockRows);
  a.cand_val = cc.cand_val;
  a.cand_id = cc.cand_id;
  a.y = static_cast<uint16_t*>(cc.y);
  a.status = cc.status;
  const int nsw = cc.bits == 2 ? plan_coarse<2>(a, max_smem, 8) : plan_coarse<4>(a, max_smem, 4);
  if (nsw < 2) return cudaErrorInvalidValue;
  if (a.NW < 1 || a.NW > kCoarseMaxWarps) return cudaErrorInvalidValue;
  if (cc.bits == 2) {
    a.dq_mul[0] = 1u << 5;   // plane 0: bits 0-1 -> 5-6
    a.dq_mul[1] = 1u << 3;   // plane 1: bits 2-3 -> 5-6
    a.dq_mul[2] = 1u << 1;   // plane 2: bits 4-5 -> 5-6
    a.dq_mul[3] = 1u << 31;  // plane 3: bits 6-7 -> 5-6 (high word of the product: >> 1)
  } else {
    a.dq_mul[0] = 1u << 3;   // low nibble: bits 0-3 -> 3-6
    a.dq_mul[1] = 1u << 31;  // high nibble: bits 4-7 -> 3-6 (>> 1)
    a.dq_mul[2] = a.dq_mul[3] = 0u;
  }
  const int grid = a.nblk < num_sms ? a.nblk : num_sms;
  const bool split = cc.bits == 4 && cc.G < 128;
  for (int m0 = 0; m0 < a.M; m0 += 8) {
    a.m0 = m0;
    a.mt = a.M - m0 < 8 ? a.M - m0 : 8;
    cudaError_t e;
    if (cc.bits == 2)
      e = launch_nsw<2, false>(a, nsw, grid, s);
    else if (split)
      e = launch_nsw<4, true>(a, nsw, grid, s);
    else
      e = launch_nsw<4, false>(a, nsw, grid, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dh
