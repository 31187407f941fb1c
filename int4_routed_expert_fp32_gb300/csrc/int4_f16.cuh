// Exact conversions of packed int4 weights and bf16 values to fp16 for the
// tensor-core expert kernels (kind::f16 MMAs on fp16 operands).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

// Two nibbles n (bits 0-3 and 16-19 of v, two's complement) -> fp16x2 q * s,
// exactly: (n ^ 8) lands in the low mantissa bits of 1024.0 (0x6400), so the
// half is 1032 + q; minus 1032 (0x6408) gives q; times the fp16 scale pair s2.
// Written in PTX with the constants as immediates (bit patterns of fp16x2).
__device__ __forceinline__ uint32_t nib_lo_f16(uint32_t v, uint32_t s2) {
  uint32_t m, r;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64086408, 0x6a;" : "=r"(m) : "r"(v));  // (v & a) ^ b
  asm("{\n .reg .b32 t;\n sub.rn.f16x2 t, %1, %2;\n mul.rn.f16x2 %0, t, %3;\n}"
      : "=r"(r)
      : "r"(m), "r"(0x64086408u), "r"(s2));
  return r;
}

// Same for nibbles at bits 4-7 and 20-23: the half is 1024 + 16 (n ^ 8);
// times 1/16 (0x2C00) minus 72 (0xD480), exact, gives q; then times s2.
__device__ __forceinline__ uint32_t nib_hi_f16(uint32_t v, uint32_t s2) {
  uint32_t m, r;
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64806480, 0x6a;" : "=r"(m) : "r"(v));
  asm("{\n .reg .b32 t;\n fma.rn.f16x2 t, %1, %2, %3;\n mul.rn.f16x2 %0, t, %4;\n}"
      : "=r"(r)
      : "r"(m), "r"(0x2C002C00u), "r"(0xD480D480u), "r"(s2));
  return r;
}

// bf16x2 -> fp16x2 (exact for values in the fp16 range; beyond it: inf).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// bf16 scale bits -> fp16 bits, replicated in both halves.
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t bf16_bits) {
  const __half h = __float2half_rn(__uint_as_float(bf16_bits << 16));
  const uint32_t u = __half_as_ushort(h);
  return u | (u << 16);
}

// Whether q * scale is exact in fp16 for every q in [-8, 7], for the two bf16
// scales of a word.  A bf16 scale m * 2^(e-7) (m the 8-bit significand)
// times q has at most 11 significant bits and its lowest set bit is at least
// 2^(e-7); fp16 holds it exactly when that bit is at least 2^-24 (e >= -17,
// exponent field >= 110) and |8 * scale| <= 65504 (e <= 12, field <= 139:
// the largest such bf16 is 8160).  Zero is exact; subnormal, infinite and
// NaN scales are not.
__device__ __forceinline__ bool scales_exact_f16(uint32_t w) {
  const uint32_t f0 = (w >> 7) & 0xFFu, f1 = (w >> 23) & 0xFFu;
  const bool z0 = (w & 0x7FFFu) == 0, z1 = (w & 0x7FFF0000u) == 0;
  return (z0 || (f0 - 110u) <= 29u) && (z1 || (f1 - 110u) <= 29u);
}

}  // namespace moe
