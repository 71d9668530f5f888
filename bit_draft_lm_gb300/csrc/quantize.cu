// Offline quantise + pack of the head weight (page "radiance_drafthead.py", _quantize_head_now):
// asymmetric min/max codes per (vocab row, group of G along K), quarter-split int2 or half-split
// int4 packing, premultiplied bf16 scale S = bf16(bias*sc) and zero term ZS = bf16(bias*sc + zp*sc).
//
// One CTA per vocab row. Every floating-point step is a separately rounded IEEE fp32 operation
// (explicit __f*_rn intrinsics, so nothing is contracted into an FMA), rounding is half-to-even
// (rintf, as torch.round), and the bf16 casts round to nearest even -- the codes and scales are
// bit-identical to the page's torch evaluation of the same formula.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dh_device.cuh"
#include "dh_launch.h"

namespace dh {

constexpr int kQuantThreads = 256;

template <int BITS>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_pack_kernel(const uint16_t* __restrict__ W, int K, int G,
                         uint8_t* __restrict__ packed, uint16_t* __restrict__ S,
                         uint16_t* __restrict__ ZS) {
  constexpr float kLevels = float((1 << BITS) - 1);
  constexpr float kBias = BITS == 2 ? 4.0f : 16.0f;  // 1 + v/4 (int2), 1 + v/16 (int4)
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int KG = K / G;
  uint16_t* w_row = reinterpret_cast<uint16_t*>(smem_raw);       // [K] bf16 bits
  float* sc_s = reinterpret_cast<float*>(smem_raw + 2 * K);        // [KG] (K*2 is 16-B aligned)
  float* zp_s = sc_s + KG;                                         // [KG]

  const int64_t n = blockIdx.x;
  const uint16_t* src = W + n * K;
  // stage the row (K % 8 == 0, 16-byte vectors)
  for (int i = threadIdx.x; i < K / 8; i += kQuantThreads)
    reinterpret_cast<uint4*>(w_row)[i] = reinterpret_cast<const uint4*>(src)[i];
  __syncthreads();

  // per-group min / max -> sc, zp (one warp per group)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int gi = warp; gi < KG; gi += kQuantThreads / 32) {
    float lo = INFINITY, hi = -INFINITY;
    for (int t = lane; t < G; t += 32) {
      const float v = bf16_bits_to_float(w_row[gi * G + t]);
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      float sc = __fdiv_rn(__fsub_rn(hi, lo), kLevels);
      if (sc < 1e-8f) sc = 1e-8f;                       // clamp(min=1e-8)
      float zp = rintf(__fdiv_rn(-lo, sc));             // round half to even
      zp = fminf(fmaxf(zp, 0.0f), kLevels);
      sc_s[gi] = sc;
      zp_s[gi] = zp;
      const float s_pre = __fmul_rn(kBias, sc);
      const float zs = __fadd_rn(s_pre, __fmul_rn(zp, sc));
      S[n * KG + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(s_pre));
      ZS[n * KG + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(zs));
    }
  }
  __syncthreads();

  auto code = [&](int k) -> uint32_t {
    const int gi = k / G;
    const float v = bf16_bits_to_float(w_row[k]);
    float q = rintf(__fadd_rn(__fdiv_rn(v, sc_s[gi]), zp_s[gi]));
    q = fminf(fmaxf(q, 0.0f), kLevels);
    return static_cast<uint32_t>(q);
  };

  // pack: 4 output bytes per thread per step (row bytes RB % 64 == 0)
  constexpr int kPlanes = 8 / BITS;  // codes per byte
  const int RB = K / kPlanes;        // bytes per row; plane p of byte j is k = p*RB + j
  uint32_t* dst = reinterpret_cast<uint32_t*>(packed + n * RB);
  for (int j4 = threadIdx.x; j4 < RB / 4; j4 += kQuantThreads) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int j = 4 * j4 + b;
      uint32_t byte = 0;
#pragma unroll
      for (int p = 0; p < kPlanes; ++p) byte |= code(p * RB + j) << (BITS * p);
      word |= byte << (8 * b);
    }
    dst[j4] = word;
  }
}

cudaError_t launch_quantize_pack(int bits, const void* W, int64_t N, int64_t K, int G,
                                 uint8_t* packed, void* S, void* ZS, cudaStream_t s) {
  const int KG = static_cast<int>(K / G);
  const size_t smem = static_cast<size_t>(2 * K) + 8 * static_cast<size_t>(KG);
  auto* Wp = static_cast<const uint16_t*>(W);
  auto* Sp = static_cast<uint16_t*>(S);
  auto* Zp = static_cast<uint16_t*>(ZS);
  cudaError_t e;
  if (bits == 2) {
    e = cudaFuncSetAttribute(quantize_pack_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    quantize_pack_kernel<2><<<static_cast<unsigned>(N), kQuantThreads, smem, s>>>(
        Wp, static_cast<int>(K), G, packed, Sp, Zp);
  } else {
    e = cudaFuncSetAttribute(quantize_pack_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    quantize_pack_kernel<4><<<static_cast<unsigned>(N), kQuantThreads, smem, s>>>(
        Wp, static_cast<int>(K), G, packed, Sp, Zp);
  }
  return cudaGetLastError();
}

}  // namespace dh
