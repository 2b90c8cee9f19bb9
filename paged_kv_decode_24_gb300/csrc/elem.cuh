// The 16-bit element types of q, K, V and out: fp16 and bf16.  Kernels take
// the type as a template parameter and convert through Elem<T>; every
// product accumulates in fp32 and the output is rounded to nearest even.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace pa {

template <typename T>
struct Elem;

template <>
struct Elem<__half> {
  // two packed elements (low first) -> fp32 pair
  static __device__ __forceinline__ float2 to_f2(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
  }
  // fp32 pair -> two packed elements, each rounded to nearest even
  static __device__ __forceinline__ uint32_t from_f2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float2 to_f2(uint32_t v) {
    // a bf16 is the top half of an fp32: widening is a shift
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  }
  static __device__ __forceinline__ uint32_t from_f2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// A pair of fp32 weights as hi + lo parts in the element type: hi is each
// value rounded to nearest even, lo the remainder (exact in fp32) rounded
// the same way.  hi + lo keeps about twice the element type's significant
// bits, so products with 16-bit operands see p to ~22 bits (fp16) or ~16
// bits (bf16) instead of 11 or 8.
template <typename T>
__device__ __forceinline__ void split_hi_lo(float2 a, uint32_t& hi, uint32_t& lo) {
  hi = Elem<T>::from_f2(a.x, a.y);
  const float2 h = Elem<T>::to_f2(hi);
  // r = a - h on both lanes with one packed fma (h * -1 + a); the
  // difference is exact in fp32
  float2 r;
  asm("{\n\t.reg .b64 ra, rh, rm, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rh, {%4, %5};\n\t"
      "mov.b64 rm, {%6, %6};\n\t"
      "fma.rn.f32x2 rd, rh, rm, ra;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(h.x), "f"(h.y), "f"(-1.f));
  lo = Elem<T>::from_f2(r.x, r.y);
}

// Eight packed elements (one 16-byte load) -> four fp32 pairs.
template <typename T>
__device__ __forceinline__ void elem8_to_float2x4(const uint4& raw, float2* f) {
  f[0] = Elem<T>::to_f2(raw.x);
  f[1] = Elem<T>::to_f2(raw.y);
  f[2] = Elem<T>::to_f2(raw.z);
  f[3] = Elem<T>::to_f2(raw.w);
}

}  // namespace pa
