// bf16 -> E4M3 codes by the rule E4M3_RNE_sat(fl32(x / d)), two elements at a time.
//
// Exact form: an IEEE fp32 division, then the hardware round-to-nearest-even
// saturating conversion; a NaN quotient gives 0x7F with the input's sign bit.
//
// Fast form, bit-identical: q = x * r with r = fl32(1 / d) is within 3 units of
// 2^-24 (relative) of x / d, and so is fl32(x / d).  Rounding to E4M3 is
// monotone, so when q * (1 - 2^-21) and q * (1 + 2^-21) round to the same code,
// the correctly rounded quotient, which lies between them, rounds to that code
// too.  Otherwise (a quotient within a few ulps of an E4M3 rounding boundary, or
// a NaN) the exact form decides.  Tiny quotients (below fp32's normal range) all
// round to a zero code either way; q overflowing to infinity only where x / d
// exceeds 448 saturates to the same code.  The fast form needs r to carry the
// relative error bound, hence the normal-range test on d.
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

// d in a range where fl32(1 / d) is a normal number with its usual error bound
__device__ __forceinline__ bool fast_ok(float d) { return fabsf(d) > 1e-30f && fabsf(d) < 1e30f; }

__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

__device__ __forceinline__ uint32_t fast_pair(uint32_t w, float r, float d) {
  const float2 q = __fmul2_rn(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)),
                              make_float2(r, r));
  const float dn = 1.0f - 0x1p-21f, up = 1.0f + 0x1p-21f;
  const float2 a = __fmul2_rn(q, make_float2(dn, dn)), b = __fmul2_rn(q, make_float2(up, up));
  const uint32_t ca = cvt_pair(a.x, a.y), cb = cvt_pair(b.x, b.y);
  // E4M3 NaN codes come only from NaN inputs (the conversion saturates): exact form
  const bool nan_code = (ca & 0x7F) == 0x7F || (ca & 0x7F00) == 0x7F00;
  if (ca == cb && !nan_code) return ca;
  return exact_pair(w, d);
}

// Eight bf16 values (one 16-byte vector) -> eight codes, low byte first.  The
// checks of fast_pair are made once per vector: the two brackets' codes are
// compared as two packed words, and NaN inputs are found on the bf16 bits
// (exponent all ones, mantissa not zero).  A vector that is not settled that
// way takes the exact form for all its elements.
__device__ __forceinline__ uint2 fast8(uint4 v, float r, float d) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const float dn = 1.0f - 0x1p-21f, up = 1.0f + 0x1p-21f;
  uint32_t lo[2] = {0, 0}, hi[2] = {0, 0};
  uint32_t nan = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 q = __fmul2_rn(make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u)),
                                make_float2(r, r));
    const float2 a = __fmul2_rn(q, make_float2(dn, dn)), b = __fmul2_rn(q, make_float2(up, up));
    lo[k >> 1] |= cvt_pair(a.x, a.y) << (16 * (k & 1));
    hi[k >> 1] |= cvt_pair(b.x, b.y) << (16 * (k & 1));
    nan |= __vcmpgtu2(w[k] & 0x7FFF7FFFu, 0x7F807F80u);
  }
  if (lo[0] == hi[0] && lo[1] == hi[1] && nan == 0) return make_uint2(lo[0], lo[1]);
  return make_uint2(exact_pair(w[0], d) | (exact_pair(w[1], d) << 16), exact_pair(w[2], d) | (exact_pair(w[3], d) << 16));
}

// Eight bf16 values -> eight codes by the fast form, settled pair by pair:
// returns a 4-bit mask of the pairs the fast form could not settle (bracket
// codes differ, or a NaN code, which only a NaN input gives); those pairs'
// codes in `out` are not final and the caller takes the exact form for them.
__device__ __forceinline__ uint32_t fast8_masked(uint4 v, float r, uint2& out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const float dn = 1.0f - 0x1p-21f, up = 1.0f + 0x1p-21f;
  uint32_t ca[4], cb[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 q = __fmul2_rn(make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u)),
                                make_float2(r, r));
    const float2 a = __fmul2_rn(q, make_float2(dn, dn)), b = __fmul2_rn(q, make_float2(up, up));
    ca[k] = cvt_pair(a.x, a.y);
    cb[k] = cvt_pair(b.x, b.y);
  }
  const uint32_t lo0 = __byte_perm(ca[0], ca[1], 0x5410), lo1 = __byte_perm(ca[2], ca[3], 0x5410);
  const uint32_t hi0 = __byte_perm(cb[0], cb[1], 0x5410), hi1 = __byte_perm(cb[2], cb[3], 0x5410);
  const uint32_t n0 = __vcmpne2((lo0 ^ hi0) | __vcmpeq4(lo0 & 0x7F7F7F7Fu, 0x7F7F7F7Fu), 0);
  const uint32_t n1 = __vcmpne2((lo1 ^ hi1) | __vcmpeq4(lo1 & 0x7F7F7F7Fu, 0x7F7F7F7Fu), 0);
  out = make_uint2(lo0, lo1);
  return (n0 & 1u) | ((n0 >> 15) & 2u) | ((n1 & 1u) << 2) | ((n1 >> 13) & 8u);
}

}  // namespace quant
}  // namespace fp8pa
