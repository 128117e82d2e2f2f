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

// Packed fp32 pairs (sm_100 family f32x2 arithmetic): each op rounds both
// halves exactly as its scalar counterpart (round to nearest, subnormals kept).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Correctly rounded x / s from r = RN(1 / s), by P. Markstein's method
// ("Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): q = RN(x r) is within 1.5 ulp;
// one correction q + r (x - s q) (residual exact with a fused multiply-add)
// makes it faithful, and by Markstein's theorem a second correction from a
// faithful quotient yields RN(x / s).  Requires a finite quotient (the callers
// bound the block maximum times r).  The residual is exact unless it underflows,
// which with s in [2^-89, 2^80] happens only for quotients below 2^-14; there the
// correction is off by less than 2^-60, far from every rounding decision of the
// target codes (the smallest, 2^-17, is E5M2's half subnormal).  The residual is
// formed as s q - x so that signed zeros keep their sign.
__device__ __forceinline__ float div_rn_markstein(float x, float s, float r) {
  float q = x * r;
  float e = fmaf(s, q, -x);
  q = fmaf(-e, r, q);
  e = fmaf(s, q, -x);
  return fmaf(-e, r, q);
}

// The same two corrections on a pair of quotients x / s.  S2 = {s, s},
// R2 = {r, r}, NR2 = {-r, -r}: -e * r is formed as e * (-r) (the same
// product), and -x as x * (-1) + (-0), exact and with the sign of zero
// flipped as a negation does.
__device__ __forceinline__ uint64_t div2_rn_markstein(uint64_t x, uint64_t S2, uint64_t R2,
                                                      uint64_t NR2) {
  const uint64_t kMinusOne = 0xBF800000BF800000ull, kMinusZero = 0x8000000080000000ull;
  const uint64_t nx = f2_fma(x, kMinusOne, kMinusZero);
  uint64_t q = f2_mul(x, R2);
  uint64_t e = f2_fma(S2, q, nx);
  q = f2_fma(e, NR2, q);
  e = f2_fma(S2, q, nx);
  return f2_fma(e, NR2, q);
}

// Two bf16 values of a word as a pair of fp32 (low element in the low half).
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// E4M3 codes of x0 / s and x1 / s (low byte from x0): the quotient is the
// correctly rounded fp32 division (corrected from rs = RN(1 / s) when `fast`,
// i.e. s in [2^-80, 2^80] and both quotients finite, else IEEE division),
// encoded to nearest, ties to even, saturating; NaN gives 0x7F with its sign.
__device__ __forceinline__ uint32_t quant2_e4m3(float x0, float x1, float s, float rs, bool fast) {
  float q0, q1;
  if (fast) {
    f2_unpack(div2_rn_markstein(f2_pack(x0, x1), f2_pack(s, s), f2_pack(rs, rs), f2_pack(-rs, -rs)),
              q0, q1);
  } else {
    q0 = x0 / s;
    q1 = x1 / s;
  }
  uint32_t c = enc2_e4m3(q0, q1);
  if (x0 != x0) c = (c & 0xFF00u) | 0x7Fu | ((__float_as_uint(x0) >> 24) & 0x80u);
  if (x1 != x1) c = (c & 0x00FFu) | ((0x7Fu | ((__float_as_uint(x1) >> 24) & 0x80u)) << 8);
  return c & 0xFFFFu;
}

}  // namespace kvq
