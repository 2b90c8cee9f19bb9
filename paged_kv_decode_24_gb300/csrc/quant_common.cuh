// Per-row quantisation of one new K or V row (the append into an 8-bit
// cache, standalone or fused into the decode kernel).
//
// INT8 rule (MonadKai/xLLM, introduction: KV-cache quantisation, per-row
// INT8): one row is one token's D-vector of one KV head; scale = max|x| / 127
// and code = x / scale rounded to nearest, ties to even, clamped to
// [-127, 127]; an all-zero row gets scale 0 and zero codes.
//
// FP8 rule ("Eine LLM-Inferenz-Engine von Grund auf mit C++ und CUDA bauen",
// section 4: FP8 quantisation of the cache): the same rows and scales with
// scale = max|x| / 448 and code = the E4M3 value nearest x / scale (ties to
// the even mantissa, magnitudes above 448 saturated to 448, the sign of a
// zero kept); E4M3 is the OCP 8-bit format with 4 exponent bits (bias 7) and
// 3 mantissa bits, largest finite 448.
//
// Both divisions are IEEE fp32 round-to-nearest (__fdiv_rn), so the codes are
// the ones any correctly rounded fp32 implementation of the rule picks.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "device_common.cuh"
#include "pa_internal.h"

namespace pa {

// Four E4M3 bytes as two half2: bytes 0, 1 into lo (byte 0 in the low half),
// bytes 2, 3 into hi.  Every E4M3 value is an fp16 value, so this is exact.
// The conversions read the register's two 16-bit halves directly.
__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two fp32 values as E4M3 bytes (a in the low byte), nearest, ties to even,
// saturated to +-448.
__device__ __forceinline__ uint32_t f2_to_e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Quantise the D fp16 values at src (global, 8-byte aligned) with one warp.
// Lane l gets the codes of dims [D/32*l, D/32*(l+1)) packed little-endian in
// the low D/32 bytes of the return value; every lane gets the scale.
template <int D, int FMT = kCodeInt8>
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
  uint32_t packed = 0;
  if constexpr (FMT == kCodeE4m3) {
    scale = __fdiv_rn(amax, 448.f);
    if (scale > 0.f) {
#pragma unroll
      for (int i = 0; i < PER; i += 2)
        packed |= f2_to_e4m3x2(__fdiv_rn(x[i], scale), __fdiv_rn(x[i + 1], scale)) << (8 * i);
    }
  } else {
    scale = __fdiv_rn(amax, 127.f);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      int c = 0;
      if (scale > 0.f) c = min(127, max(-127, __float2int_rn(__fdiv_rn(x[i], scale))));
      packed |= (uint32_t)(c & 0xff) << (8 * i);
    }
  }
  return packed;
}

}  // namespace pa
