// kvq_codecs.cuh -- device encode/decode of the cache formats (sm_103a).
//
// Formats: "Quantized KV Cache" (SGLang documentation), Supported formats:
// FP8 E4M3 / E5M2, FP4 E2M1 with a shared 8-bit exponent per 16 elements;
// "SGLang PR #21954 analysis: NVFP4 KV cache", Code analysis 1: NVFP4 = fp32
// per-tensor scale x FP8-E4M3 per-block scale x E2M1.  Conversions use the
// PTX cvt instructions for these types (round to nearest even, satfinite).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace kvq {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Two fp32 -> two E4M3fn codes (low byte from `lo`), RNE, saturating.
__device__ __forceinline__ uint32_t enc2_e4m3(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t enc2_e5m2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two fp32 -> one byte of two E2M1 codes (low nibble from `lo`).
__device__ __forceinline__ uint32_t enc2_e2m1(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 / E5M2 codes (low 16 bits of x) -> half2 (exact).
__device__ __forceinline__ uint32_t dec2_e4m3_h2(uint32_t x) {
  uint32_t r;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, l; }" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t dec2_e4m3_h2_hi(uint32_t x) {
  uint32_t r;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, h; }" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t dec2_e5m2_h2(uint32_t x) {
  uint32_t r;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e5m2x2 %0, l; }" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t dec2_e5m2_h2_hi(uint32_t x) {
  uint32_t r;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e5m2x2 %0, h; }" : "=r"(r) : "r"(x));
  return r;
}
// Byte `B` of x (two E2M1 codes) -> half2 (exact; low half from the low nibble).
template <int B>
__device__ __forceinline__ uint32_t dec2_e2m1_h2(uint32_t x) {
  uint32_t r;
  if (B == 0)
    asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b0; }"
        : "=r"(r) : "r"(x));
  else if (B == 1)
    asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b1; }"
        : "=r"(r) : "r"(x));
  else if (B == 2)
    asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b2; }"
        : "=r"(r) : "r"(x));
  else
    asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b3; }"
        : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ float h2_lo(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFF)));
}
__device__ __forceinline__ float h2_hi(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)(h >> 16)));
}

// Exact fp32 value of one E4M3 code.
__device__ __forceinline__ float dec_e4m3(uint32_t code) { return h2_lo(dec2_e4m3_h2(code & 0xFF)); }

// Exact fp32 value of an E8M0 byte: 2^(c - 127) (c = 0 is the subnormal 2^-127).
__device__ __forceinline__ float dec_e8m0(uint32_t c) {
  c &= 0xFF;
  if (c == 0xFF) return __uint_as_float(0x7FC00000u);
  return c == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(c << 23);
}

// 2^n as fp32 for n in [-127, 127] (exact; 2^-127 is subnormal).
__device__ __forceinline__ float exp2i(int n) {
  return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23) : __uint_as_float(0x00400000u);
}

// floor(log2(a)) for a finite a > 0, from the fp32 bits (handles subnormals).
__device__ __forceinline__ int floor_log2(float a) {
  uint32_t b = __float_as_uint(a);
  int e = (int)((b >> 23) & 0xFF);
  if (e != 0) return e - 127;
  uint32_t m = b & 0x7FFFFF;
  return -149 + (31 - __clz(m));
}

// bfloat16 round-to-nearest-even of an fp32 value; NaN -> 0x7FC0.
__device__ __forceinline__ uint32_t bf16_rne_bits(float x) {
  if (x != x) return 0x7FC0u;
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

}  // namespace kvq
