// Offline quantise + pack of the head weight (page "radiance_drafthead.py", the load-time quantiser):
// asymmetric min/max codes per (vocab row, group of G along K), quarter-split int2 or half-split
// int4 packing, premultiplied bf16 scale S = bf16(bias*sc) and zero term ZS = bf16(bias*sc + zp*sc).
//
// Input rows are bf16, or (FP8 checkpoints, the page's FP8 head) e4m3 bytes with an fp32
// per-row scale: w = e4m3(b) * scale[n], one fp32 multiply, as the page's `wg * wsc[i:j, None]`.
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

template <int BITS, bool FP8>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_pack_kernel(const void* __restrict__ W, const float* __restrict__ row_scale, int K,
                         int G, uint8_t* __restrict__ packed, uint16_t* __restrict__ S,
                         uint16_t* __restrict__ ZS) {
  constexpr float kLevels = float((1 << BITS) - 1);
  constexpr float kBias = BITS == 2 ? 4.0f : 16.0f;  // 1 + v/4 (int2), 1 + v/16 (int4)
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int KG = K / G;
  float* w_row = reinterpret_cast<float*>(smem_raw);  // [K] the row's values (exact in fp32)
  float* sc_s = w_row + K;                            // [KG]
  float* zp_s = sc_s + KG;                            // [KG]

  const int64_t n = blockIdx.x;
  // stage the row (K % 8 == 0, 16-byte vectors of bf16, 8-byte vectors of e4m3)
  if (FP8) {
    const float rs = row_scale[n];
    const uint2* src = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(W) + n * K);
    for (int i = threadIdx.x; i < K / 8; i += kQuantThreads) {
      const uint2 v = src[i];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint32_t byte = ((b < 4 ? v.x : v.y) >> (8 * (b & 3))) & 0xffu;
        w_row[8 * i + b] = __fmul_rn(e4m3_bits_to_f32(byte), rs);
      }
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(W) + n * K);
    for (int i = threadIdx.x; i < K / 8; i += kQuantThreads) {
      const uint4 v = src[i];
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        w_row[8 * i + 2 * b] = bf16_bits_to_float(w4[b] & 0xffffu);
        w_row[8 * i + 2 * b + 1] = bf16_bits_to_float(w4[b] >> 16);
      }
    }
  }
  __syncthreads();

  // per-group min / max -> sc, zp (one warp per group)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int gi = warp; gi < KG; gi += kQuantThreads / 32) {
    float lo = INFINITY, hi = -INFINITY;
    for (int t = lane; t < G; t += 32) {
      const float v = w_row[gi * G + t];
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
    const float v = w_row[k];
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

template <int BITS, bool FP8>
static cudaError_t launch_qp(const void* W, const float* row_scale, int64_t N, int64_t K, int G,
                             uint8_t* packed, uint16_t* S, uint16_t* ZS, cudaStream_t s) {
  const size_t smem = 4 * static_cast<size_t>(K) + 8 * static_cast<size_t>(K / G);
  const cudaError_t e = cudaFuncSetAttribute(quantize_pack_kernel<BITS, FP8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  quantize_pack_kernel<BITS, FP8><<<static_cast<unsigned>(N), kQuantThreads, smem, s>>>(
      W, row_scale, static_cast<int>(K), G, packed, S, ZS);
  return cudaGetLastError();
}

cudaError_t launch_quantize_pack(int bits, const void* W, int64_t N, int64_t K, int G,
                                 uint8_t* packed, void* S, void* ZS, cudaStream_t s,
                                 const float* row_scale) {
  auto* Sp = static_cast<uint16_t*>(S);
  auto* Zp = static_cast<uint16_t*>(ZS);
  if (row_scale != nullptr)
    return bits == 2 ? launch_qp<2, true>(W, row_scale, N, K, G, packed, Sp, Zp, s)
                     : launch_qp<4, true>(W, row_scale, N, K, G, packed, Sp, Zp, s);
  return bits == 2 ? launch_qp<2, false>(W, nullptr, N, K, G, packed, Sp, Zp, s)
                   : launch_qp<4, false>(W, nullptr, N, K, G, packed, Sp, Zp, s);
}

}  // namespace dh
