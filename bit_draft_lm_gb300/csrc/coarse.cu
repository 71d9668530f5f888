// Host side of the coarse pass: shared-memory plan and dispatch to the kernel instantiations
// (coarse_i2g128.cu, coarse_i2g64.cu, coarse_i4g128.cu, coarse_i4g64.cu).
#include <cuda_runtime.h>

#include "coarse_kernel.cuh"
#include "dh_launch.h"

namespace dh {

cudaError_t launch_coarse_i2g128(const CoarseArgs& a, int nsw, int grid, cudaStream_t s);
cudaError_t launch_coarse_i2g64(const CoarseArgs& a, int nsw, int grid, cudaStream_t s);
cudaError_t launch_coarse_i4g128(const CoarseArgs& a, int nsw, int grid, cudaStream_t s);
cudaError_t launch_coarse_i4g64(const CoarseArgs& a, int nsw, int grid, cudaStream_t s);

// Shared-memory plan for one launch; returns the weight ring depth (0 if nothing fits).
// mt_cap: most hidden rows per pass (8, or fewer when the partial buffers of 8 do not fit).
template <int BITS>
static int plan_coarse(CoarseArgs& a, int max_smem, int nsw_max, int mt_cap) {
  constexpr int SB = BITS == 2 ? 64 : 128;
  a.RB = a.K * BITS / 8;
  a.KG = a.K / a.G;
  a.NW = a.K / 256;
  const int mt_max = a.M < mt_cap ? a.M : mt_cap;
  a.red_pitch = mt_max | 1;  // odd: a warp reading one column over 32 rows hits 32 banks
  const int red_buf = (a.NW + 1) * kBlockRows * a.red_pitch * 4;  // NW warps + zero-point slot
  const int wstage = kTileRows * SB;
  // {ring depth, partial buffers, S/ZS block stages}, first that fits. A 4-deep ring (3 tiles in
  // flight per warp, 60 KB per SM) measured faster than an 8-deep one at one hidden row on
  // GB300 (51.3 vs 53.5 us): the deeper initial burst delays every warp's first tile. Two S/ZS
  // stages make room for 8 hidden rows of the int4 head and of 64-wide groups at K = 5120.
  static const int kPlans[][3] = {{4, 4, 4}, {8, 4, 4}, {8, 2, 4}, {4, 2, 4}, {4, 2, 2},
                                  {2, 2, 4}, {2, 2, 2}};
  for (const auto& pl : kPlans) {
    const int nsw = pl[0], nb = pl[1], nsb = pl[2];
    if (nsw > nsw_max) continue;
    int off = 0;
    a.off_bars = off;
    off += (kSBlocks + kMaxRedBufs) * 8 + (3 * kMaxRedBufs + kSBlocks + 2) * 4 + 16;
    a.off_xs = off = (off + 15) / 16 * 16;
    off += a.NW * 8 * 4 * 4;   // strip group sums: [NW][8 rows][<= 4 groups] fp32
    off += mt_max * a.KG * 4;  // group sums of the row: [mt][K/G] fp32
    a.off_zb = off = (off + 15) / 16 * 16;
    off += (a.KG / 8) * 3 * mt_max * 4 * 8;  // zero-point MMA B fragments: [K/G/8][3][mt][4] uint2
    a.off_sz = off = (off + 127) / 128 * 128;
    off += nsb * 2 * kBlockRows * a.KG * 2;
    a.off_red = off = (off + 15) / 16 * 16;
    const int ring = (a.off_red + nb * red_buf + 127) / 128 * 128;
    if (ring + a.NW * nsw * wstage <= max_smem) {
      a.nb = nb;
      a.nsb = nsb;
      a.nsb_log = nsb == 4 ? 2 : 1;
      a.off_ring = ring;
      return nsw;
    }
  }
  return 0;
}

// Returns cudaErrorInvalidValue if the shape does not fit the kernel's plan.
cudaError_t launch_coarse_topk(const CoarseCall& cc, int num_sms, int max_smem, cudaStream_t s) {
  // many hidden rows of an int2 head: one tensor-core pass instead of several warp-MMA passes
  if (cc.scratch != nullptr && coarse_wide_supports(cc))
    return launch_coarse_wide(cc, cc.scratch, num_sms, max_smem, s);
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
  if (cc.G != 64 && cc.G != 128) return cudaErrorInvalidValue;
  // passes of 8 hidden rows (one MMA column tile); where their partial buffers do not fit next
  // to the rings (the int4 head with 64-wide groups at K = 5120), passes of 4, 2 or 1
  int nsw = 0, pass_rows = 8;
  for (; pass_rows >= 1; pass_rows /= 2) {
    nsw = cc.bits == 2 ? plan_coarse<2>(a, max_smem, 8, pass_rows)
                       : plan_coarse<4>(a, max_smem, 4, pass_rows);
    if (nsw >= 2) break;
  }
  if (nsw < 2) return cudaErrorInvalidValue;
  if (a.NW < 1 || a.NW > kCoarseMaxWarps || a.KG % 8) return cudaErrorInvalidValue;
  a.u16_mul = 1u << 16;
  const int grid = a.nblk < num_sms ? a.nblk : num_sms;
  for (int m0 = 0; m0 < a.M; m0 += pass_rows) {
    a.m0 = m0;
    a.mt = a.M - m0 < pass_rows ? a.M - m0 : pass_rows;
    cudaError_t e;
    if (cc.bits == 2)
      e = cc.G == 128 ? launch_coarse_i2g128(a, nsw, grid, s) : launch_coarse_i2g64(a, nsw, grid, s);
    else
      e = cc.G == 128 ? launch_coarse_i4g128(a, nsw, grid, s) : launch_coarse_i4g64(a, nsw, grid, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dh
