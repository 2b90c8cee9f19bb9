// Per-row INT8 quantisation of one new K or V row (the append into the INT8
// cache, standalone or fused into the decode kernel).
//
// Rule (MonadKai/xLLM, introduction: KV-cache quantisation, per-row INT8):
// one row is one token's D-vector of one KV head; scale = max|x| / 127 and
// code = x / scale rounded to nearest, ties to even, clamped to [-127, 127];
// an all-zero row gets scale 0 and zero codes.  Both divisions are IEEE fp32
// round-to-nearest (__fdiv_rn), so the codes are the ones any correctly
// rounded fp32 implementation of the rule picks.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "device_common.cuh"

namespace pa {

// Quantise the D fp16 values at src (global, 8-byte aligned) with one warp.
// Lane l gets the codes of dims [D/32*l, D/32*(l+1)) packed little-endian in
// the low D/32 bytes of the return value; every lane gets the scale.
template <int D>
__device__ __forceinline__ uint32_t quantize_row_warp(const __half* src, int lane, float& scale) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  constexpr int PER = D / 32;
  float x[PER];
  if constexpr (PER == 4) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(src) + lane);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    x[0] = a.x;
    x[1] = a.y;
    x[2] = b.x;
    x[3] = b.y;
  } else {
    const uint32_t raw = __ldg(reinterpret_cast<const unsigned int*>(src) + lane);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw));
    x[0] = a.x;
    x[1] = a.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
  scale = __fdiv_rn(amax, 127.f);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    int c = 0;
    if (scale > 0.f) c = min(127, max(-127, __float2int_rn(__fdiv_rn(x[i], scale))));
    packed |= (uint32_t)(c & 0xff) << (8 * i);
  }
  return packed;
}

}  // namespace pa
