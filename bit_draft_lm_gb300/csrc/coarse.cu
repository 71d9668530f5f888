// Coarse pass + block top-KCAND of the low-bit draft head (page "radiance_drafthead.py":
// module docstring, _draft_head_int2 and _emit), for sm_103a.
//
// Work decomposition (GB300-first, not the page's one-program-per-block grid):
//  * Persistent grid, one CTA per SM. A CTA walks 64-row candidate blocks b = blockIdx.x,
//    blockIdx.x + gridDim.x, ...; each block is four 16-row tiles.
//  * One producer warp streams every tile (16 packed rows + their S and ZS rows) into a ring of
//    shared-memory stages with 1-D bulk copies (TMA engine, mbarrier completion). Packed rows
//    land at a pitch of 64 (mod 128) bytes so the consumers' 16-byte reads are conflict-free.
//  * NW = K/256 consumer warps. Warp w owns the same 256 k-values of every row ("strip": bytes
//    [64w, 64w+64) of each int2 row, [128w, 128w+128) of each int4 row), so its share of the
//    hidden states never changes: the permuted x fragments of the MMA's B operand are loaded
//    into registers once per launch and the kernel reads no x from shared memory in its loop.
//  * Per tile a warp dequantises its strip with the page's bit patterns straight into MMA A
//    fragments (0x3F80 | ((b << (5-2q)) & 0x60) = 1 + v/4 for int2, 0x3F80 | (nibble << 3) =
//    1 + v/16 for int4; weights on the MMA's 16-row side, hidden rows on its 8-column side) and
//    issues mma.sync m16n8k16 (bf16 in, fp32 accumulate). The MMA's k order is permuted so that
//    byte j and byte j+2 of a 32-bit word share one bf16x2 register; x is permuted the same way.
//  * The per-group scale is applied to the accumulator, never to the weight tile:
//    acc += S[n,g] * P_g per (plane, strip) and acc -= sum_g ZS[n,g] * XS[m,g] once per tile as a
//    short MMA whose B operand is -XS split into three bf16 parts (K' = 3*K/G, padded to 16).
//  * Block epilogue: partial accumulators of the NW warps are summed in a fixed order (the
//    result does not depend on timing), then warp m selects the KCAND largest of the block's 64
//    coarse values for hidden row m with warp reductions (max key, then lowest row on ties).
// Hidden rows are processed eight at a time (one MMA column tile); M > 8 runs ceil(M/8) passes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dh_device.cuh"
#include "dh_launch.h"

namespace dh {

constexpr int kCoarseMaxWarps = 20;                  // K <= 5120
constexpr int kCoarseMaxThreads = (kCoarseMaxWarps + 1) * 32;
constexpr int kBlkPitch = 9;                         // floats per row of the block value table

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
  // shared-memory layout (bytes)
  int pitch, stage_bytes, s_off, zs_off, nstages;
  int off_red, off_xsfrag, off_xs, off_blk, off_bars, off_stages;
};

// int2: bf16x2 of plane q for the even bytes (b0, b2) or odd bytes (b1, b3) of word w.
__device__ __forceinline__ uint32_t deq2(uint32_t w, int q, bool odd) {
  uint32_t t;
  if (odd) {
    t = w >> (3 + 2 * q);
  } else {
    t = q < 3 ? (w << (5 - 2 * q)) : (w >> 1);
  }
  return (t & 0x00600060u) | 0x3F803F80u;  // 1 + v/4
}
// int4: nibble h.
__device__ __forceinline__ uint32_t deq4(uint32_t w, int h, bool odd) {
  uint32_t t;
  if (odd) {
    t = w >> (5 + 4 * h);
  } else {
    t = h == 0 ? (w << 3) : (w >> 1);
  }
  return (t & 0x00780078u) | 0x3F803F80u;  // 1 + v/16
}

template <int BITS>
__device__ __forceinline__ uint32_t deq(uint32_t w, int p, bool odd) {
  return BITS == 2 ? deq2(w, p, odd) : deq4(w, p, odd);
}

// SPLIT: the strip spans more than one quantisation group per plane (int4 with G = 64), so the
// accumulator is folded once per 64-byte sub-chunk instead of once per strip.
template <int BITS, bool SPLIT>
__global__ void __launch_bounds__(kCoarseMaxThreads, 1) coarse_topk_kernel(const CoarseArgs a) {
  constexpr int P = 8 / BITS;   // codes per byte (planes)
  constexpr int SB = 256 / P;   // strip bytes per warp: 256 k-values
  constexpr int U = SB / 64;    // 64-byte sub-chunks per strip
  constexpr int FS = SPLIT ? U : 1;
  extern __shared__ __align__(128) unsigned char sm[];

  const int NW = a.NW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + a.off_bars);
  uint64_t* empty = full + a.nstages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + a.nstages);
  const int NS = a.nstages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], static_cast<uint32_t>(NW));
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  // ------------------------------------------------------------------ producer warp
  if (warp == NW) {
    if (lane == 0) {
      uint32_t it = 0;
      bool aborted = false;
      for (int b = blockIdx.x; b < a.nblk && !aborted; b += gridDim.x) {
        for (int t = 0; t < kTilesPerBlock; ++t) {
          const int s = static_cast<int>(it % NS);
          const uint32_t use = it / NS;
          if (use > 0 && !mbar_wait_bounded(&empty[s], (use - 1) & 1u)) {
            *abort_flag = 1;
            set_status(a.status, DH_DEV_WAIT_TIMEOUT);
            aborted = true;
            break;
          }
          if (*abort_flag) {
            aborted = true;
            break;
          }
          const int row0 = b * kBlockRows + t * kTileRows;
          int nv = a.N - row0;
          nv = nv < 0 ? 0 : (nv > kTileRows ? kTileRows : nv);
          unsigned char* st = sm + a.off_stages + s * a.stage_bytes;
          const uint32_t sbytes = static_cast<uint32_t>(nv * a.KG * 2);
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nv * a.RB) + 2u * sbytes);
          for (int r = 0; r < nv; ++r)
            bulk_g2s(st + r * a.pitch, a.packed + static_cast<int64_t>(row0 + r) * a.RB,
                     static_cast<uint32_t>(a.RB), &full[s]);
          if (nv > 0) {
            bulk_g2s(st + a.s_off, a.S + static_cast<int64_t>(row0) * a.KG, sbytes, &full[s]);
            bulk_g2s(st + a.zs_off, a.ZS + static_cast<int64_t>(row0) * a.KG, sbytes, &full[s]);
          }
          ++it;
        }
      }
      // never leave the CTA with copies in flight: wait for the last use of every stage
      const uint32_t first = it > static_cast<uint32_t>(NS) ? it - NS : 0u;
      for (uint32_t k = first; k < it; ++k)
        if (!mbar_wait_bounded(&full[k % NS], (k / NS) & 1u))
          set_status(a.status, DH_DEV_WAIT_TIMEOUT);
    }
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  const int nthr = NW * 32;
  const int KG = a.KG;
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
          const int k0 = p * (a.K / P) + warp * SB + 64 * u + 16 * c + 4 * i;
          const uint2 v = *reinterpret_cast<const uint2*>(
              a.x + static_cast<int64_t>(a.m0 + g) * a.K + k0);
          b0 = __byte_perm(v.x, v.y, 0x5410);  // (x[k0], x[k0+2]): even bytes of the word
          b1 = __byte_perm(v.x, v.y, 0x7632);  // (x[k0+1], x[k0+3]): odd bytes
        }
        bfr[u][i][p][0] = b0;
        bfr[u][i][p][1] = b1;
      }

  // group sums of x (fp32) -> -XS as bf16 hi + lo B fragments of the ZS term
  float* xs_s = reinterpret_cast<float*>(sm + a.off_xs);  // [8][KG]
  for (int pr = warp; pr < a.mt * KG; pr += NW) {
    const int tok = pr / KG, gi = pr - tok * KG;
    const uint16_t* xr = a.x + static_cast<int64_t>(a.m0 + tok) * a.K + gi * a.G;
    float sum = 0.0f;
    for (int t = lane; t < a.G; t += 32) sum += bf16_bits_to_float(xr[t]);
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) xs_s[tok * KG + gi] = sum;
  }
  named_bar_sync(1, nthr);
  // -XS as three bf16 parts (hi + mid + lo, relative error 2^-27): virtual column vk of the ZS
  // term's MMA is part vk / KG of group vk % KG; columns past 3*KG are zero padding.
  const int zs_steps = (3 * KG + 15) / 16;
  uint2* xsfrag = reinterpret_cast<uint2*>(sm + a.off_xsfrag);  // [zs_steps][32]
  for (int e = threadIdx.x; e < zs_steps * 32; e += nthr) {
    const int ks = e >> 5, l = e & 31, gg = l >> 2, cc = l & 3;
    uint32_t h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int vk = 16 * ks + 2 * cc + (q & 1) + (q >> 1) * 8;
      const int part = vk / KG, gi = vk - part * KG;
      float v = (gg < a.mt && part < 3) ? xs_s[gg * KG + gi] : 0.0f;
      __nv_bfloat16 pv = __float2bfloat16_rn(v);
      for (int t = 0; t < part; ++t) {  // peel off the parts above this one
        v -= __bfloat162float(pv);
        pv = __float2bfloat16_rn(v);
      }
      h[q] = static_cast<uint32_t>(__bfloat16_as_ushort(pv)) ^ 0x8000u;  // -XS part
    }
    xsfrag[e] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  }
  named_bar_sync(1, nthr);

  float4* red = reinterpret_cast<float4*>(sm + a.off_red);  // [NW][4 tiles][32 lanes]
  float* blk = reinterpret_cast<float*>(sm + a.off_blk);    // [64 rows][kBlkPitch]
  const int strip_byte = warp * SB;

  uint32_t it = 0;
  for (int b = blockIdx.x; b < a.nblk; b += gridDim.x) {
#pragma unroll 1
    for (int t = 0; t < kTilesPerBlock; ++t) {
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const int s = static_cast<int>(it % NS);
      const uint32_t use = it / NS;
      ++it;
      if (!*abort_flag && !mbar_wait_bounded(&full[s], use & 1u)) {
        *abort_flag = 1;
        set_status(a.status, DH_DEV_WAIT_TIMEOUT);
      }
      const unsigned char* st = sm + a.off_stages + s * a.stage_bytes;
      const unsigned char* rg = st + g * a.pitch + strip_byte + 16 * c;
      const unsigned char* rg8 = rg + 8 * a.pitch;
      float d[FS][P][4];
#pragma unroll
      for (int f = 0; f < FS; ++f)
#pragma unroll
        for (int p = 0; p < P; ++p)
#pragma unroll
          for (int e = 0; e < 4; ++e) d[f][p][e] = 0.0f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint4 wa = *reinterpret_cast<const uint4*>(rg + 64 * u);
        const uint4 wb = *reinterpret_cast<const uint4*>(rg8 + 64 * u);
        const uint32_t wav[4] = {wa.x, wa.y, wa.z, wa.w};
        const uint32_t wbv[4] = {wb.x, wb.y, wb.z, wb.w};
        const int f = SPLIT ? u : 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int p = 0; p < P; ++p)
            mma_bf16_16816(d[f][p], deq<BITS>(wav[i], p, false), deq<BITS>(wbv[i], p, false),
                           deq<BITS>(wav[i], p, true), deq<BITS>(wbv[i], p, true),
                           bfr[u][i][p][0], bfr[u][i][p][1], d[f][p]);
      }
      // scale on the accumulator: acc += S[n, g] * P_g
      const uint16_t* Sst = reinterpret_cast<const uint16_t*>(st + a.s_off);
#pragma unroll
      for (int f = 0; f < FS; ++f)
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const int gi = p * (a.RB / a.G) + (strip_byte + 64 * f) / a.G;
          const float sg = bf16_bits_to_float(Sst[g * KG + gi]);
          const float sg8 = bf16_bits_to_float(Sst[(g + 8) * KG + gi]);
          acc[0] = fmaf(sg, d[f][p][0], acc[0]);
          acc[1] = fmaf(sg, d[f][p][1], acc[1]);
          acc[2] = fmaf(sg8, d[f][p][2], acc[2]);
          acc[3] = fmaf(sg8, d[f][p][3], acc[3]);
        }
      // zero-point term once per tile: acc -= sum_g ZS[n, g] * XS[m, g]
      if (warp == (t * NW) / kTilesPerBlock) {
        const unsigned char* zst = st + a.zs_off;
        const int lr = (lane & 7) + ((lane >> 3) & 1) * 8;
        for (int ks = 0; ks < zs_steps; ++ks) {
          const int col = (16 * ks + 8 * (lane >> 4)) % KG;  // B is zero past 3*KG
          uint32_t z0, z1, z2, z3;
          ldmatrix_x4(z0, z1, z2, z3, zst + (lr * KG + col) * 2);
          const uint2 xb = xsfrag[ks * 32 + lane];
          mma_bf16_16816(acc, z0, z1, z2, z3, xb.x, xb.y, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      red[(warp * kTilesPerBlock + t) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }

    // ---- block epilogue: fixed-order sum of the warps' partials, then top-KCAND per row
    named_bar_sync(1, nthr);
    if (threadIdx.x < kTilesPerBlock * 32) {
      const int t = threadIdx.x >> 5, L = threadIdx.x & 31;
      float4 sum = red[t * 32 + L];
      for (int w = 1; w < NW; ++w) {
        const float4 v = red[(w * kTilesPerBlock + t) * 32 + L];
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
      }
      const int gg = L >> 2, cc = L & 3;
      const int ra = t * kTileRows + gg, rb = ra + 8;
      blk[ra * kBlkPitch + 2 * cc] = sum.x;
      blk[ra * kBlkPitch + 2 * cc + 1] = sum.y;
      blk[rb * kBlkPitch + 2 * cc] = sum.z;
      blk[rb * kBlkPitch + 2 * cc + 1] = sum.w;
      if (a.y) {
        const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = b * kBlockRows + ((e >> 1) ? rb : ra);
          const int tok = 2 * cc + (e & 1);
          if (row < a.N && tok < a.mt)
            a.y[static_cast<int64_t>(a.m0 + tok) * a.N + row] =
                __bfloat16_as_ushort(__float2bfloat16_rn(vals[e]));
        }
      }
    }
    named_bar_sync(1, nthr);
    for (int m = warp; m < a.mt; m += NW) {
      const int n0 = b * kBlockRows + lane;
      uint32_t k0 = n0 < a.N ? order_key(blk[lane * kBlkPitch + m]) : 0u;
      uint32_t k1 = n0 + 32 < a.N ? order_key(blk[(lane + 32) * kBlkPitch + m]) : 0u;
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
  }
}


// Shared-memory plan for one launch; returns false if it does not fit.
static bool plan_coarse(CoarseArgs& a, int bits, int max_smem) {
  a.RB = static_cast<int>(a.K * bits / 8);
  a.KG = a.K / a.G;
  a.NW = a.K / 256;
  a.pitch = (a.RB % 128 == 0) ? a.RB + 64 : a.RB;  // 64 (mod 128): conflict-free 16-B reads
  a.s_off = kTileRows * a.pitch;
  a.zs_off = a.s_off + kTileRows * a.KG * 2;
  a.stage_bytes = a.zs_off + kTileRows * a.KG * 2;
  int off = 0;
  a.off_red = off;
  off += a.NW * kTilesPerBlock * 32 * 16;
  a.off_xsfrag = off;
  off += ((3 * a.KG + 15) / 16) * 32 * 8;
  a.off_xs = off;
  off += 8 * a.KG * 4;
  a.off_blk = off;
  off += ((kBlockRows * kBlkPitch * 4 + 15) / 16) * 16;
  a.off_bars = off;
  const int fixed_wo_bars = off;
  // stages: as many as fit, up to 8
  int ns = 8;
  for (; ns >= 2; --ns) {
    int bars = 2 * ns * 8 + 16;
    int stages_at = ((fixed_wo_bars + bars + 127) / 128) * 128;
    if (stages_at + ns * a.stage_bytes <= max_smem) break;
  }
  if (ns < 2) return false;
  a.nstages = ns;
  a.off_stages = ((fixed_wo_bars + 2 * ns * 8 + 16 + 127) / 128) * 128;
  return true;
}

static int smem_total(const CoarseArgs& a) { return a.off_stages + a.nstages * a.stage_bytes; }

template <int BITS, bool SPLIT>
static cudaError_t launch_one(const CoarseArgs& a, int grid, cudaStream_t s) {
  const int smem = smem_total(a);
  cudaError_t e = cudaFuncSetAttribute(coarse_topk_kernel<BITS, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  coarse_topk_kernel<BITS, SPLIT><<<grid, (a.NW + 1) * 32, smem, s>>>(a);
  return cudaGetLastError();
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
  if (!plan_coarse(a, cc.bits, max_smem)) return cudaErrorInvalidValue;
  if (a.NW < 1 || a.NW > kCoarseMaxWarps) return cudaErrorInvalidValue;
  const int grid = a.nblk < num_sms ? a.nblk : num_sms;
  const bool split = cc.bits == 4 && cc.G < 128;
  for (int m0 = 0; m0 < a.M; m0 += 8) {
    a.m0 = m0;
    a.mt = a.M - m0 < 8 ? a.M - m0 : 8;
    cudaError_t e;
    if (cc.bits == 2)
      e = launch_one<2, false>(a, grid, s);
    else if (split)
      e = launch_one<4, true>(a, grid, s);
    else
      e = launch_one<4, false>(a, grid, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dh
