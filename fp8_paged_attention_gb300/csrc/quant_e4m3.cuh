// bf16 -> E4M3 codes by the rule E4M3_RNE_sat(fl32(x / d)), eight elements at a time.
//
// Exact form: an IEEE fp32 division, then the hardware round-to-nearest-even
// saturating conversion; a NaN quotient gives 0x7F with the input's sign bit.
//
// Fast form, bit-identical: the correctly rounded quotient fl32(x / d) without a
// division, by Markstein's correction (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1),
// 1990; also Muller et al., Handbook of Floating-Point Arithmetic, the section
// on division with a fused multiply-add).  With y = RN(1 / d) and q a faithful
// rounding of x / d, the residual r = x - d * q is exact in fp32 and
// RN(q + r * y) = RN(x / d).  The start q0 = RN(x * y) lies within 2^-23
// (relative) of x / d; one correction step from it forms q0 + r0 * y within
// 2^-46 of x / d before its one rounding, so its result is faithful, and the
// second step is Markstein's.  Each residual and each correction is one fused
// multiply-add (one rounding).
//
// Range: 2^-64 <= d <= 2^64.  A quotient below 2^-11 gives a zero code whatever
// the steps do to it (the smallest E4M3 rounding boundary is 2^-10, and they move
// it by far less than that); for a larger quotient every residual the steps need
// has its last bit at or above 2^-121, so none is lost to underflow.  The code's
// sign is the input's (d > 0), which keeps -0 right.  An infinite input, or a
// product x * y that overflows, makes the steps give NaN: those codes, and NaN
// inputs, show as the NaN code 0x7F and are flagged for the exact form.
#pragma once
#include <cuda_fp8.h>
#include <stdint.h>

namespace fp8pa {
namespace quant {

__device__ __forceinline__ uint32_t exact_one(uint16_t bits, float d) {
  const float v = __fdiv_rn(__uint_as_float((uint32_t)bits << 16), d);
  if (v != v) return (uint32_t)(0x7F | ((bits >> 8) & 0x80));
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Two bf16 values (low half first) -> two codes (low byte first).
__device__ __forceinline__ uint32_t exact_pair(uint32_t w, float d) {
  return exact_one((uint16_t)w, d) | (exact_one((uint16_t)(w >> 16), d) << 8);
}

// d in the range where the fast form is exact
__device__ __forceinline__ bool fast_ok(float d) { return d >= 0x1p-64f && d <= 0x1p64f; }

__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

// Eight bf16 values (one 16-byte vector) -> eight codes by the fast form, low
// byte first; y = RN(1 / d), nd = -d, d in the fast_ok range.  `flags` gets
// 0x80 in each byte whose code is the NaN code: the caller takes the exact form
// for those (they come only from NaN or infinite inputs or an overflowing x * y).
__device__ __forceinline__ uint2 fast8(uint4 v, float y, float nd, uint2& flags) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const float2 y2 = make_float2(y, y), nd2 = make_float2(nd, nd);
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
    float2 q = __fmul2_rn(x, y2);
#pragma unroll
    for (int s = 0; s < 2; ++s) q = __ffma2_rn(__ffma2_rn(q, nd2, x), y2, q);  // q += (x - d q) y
    c[k] = cvt_pair(q.x, q.y);
  }
  const uint32_t mag = 0x7F7F7F7Fu;
  const uint32_t c0 = __byte_perm(c[0], c[1], 0x5410) & mag, c1 = __byte_perm(c[2], c[3], 0x5410) & mag;
  // (b & 0x7F) + 1 sets bit 7 of a byte exactly when its code is 0x7F / 0xFF
  flags = make_uint2((c0 + 0x01010101u) & ~mag, (c1 + 0x01010101u) & ~mag);
  // sign bits of the eight inputs: bit 15 and bit 31 of each word
  const uint32_t s0 = __byte_perm(w[0], w[1], 0x7531), s1 = __byte_perm(w[2], w[3], 0x7531);
  return make_uint2(c0 | (s0 & ~mag), c1 | (s1 & ~mag));
}

// The pairs (input words) of a vector whose codes `fast8` flagged: bit j for word j.
__device__ __forceinline__ uint32_t flagged_pairs(uint2 f) {
  return (uint32_t)((f.x & 0x8080u) != 0) | ((uint32_t)((f.x >> 16) != 0) << 1) |
         ((uint32_t)((f.y & 0x8080u) != 0) << 2) | ((uint32_t)((f.y >> 16) != 0) << 3);
}

}  // namespace quant
}  // namespace fp8pa
