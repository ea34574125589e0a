// Software 2^x for a pair of floats on the FMA and integer pipes, the way
// FA4 offloads part of the softmax's exponentials from the MUFU unit
// ("FlashAttention: Part 2", sections 1.7 and 1.8: the exponential is the
// Blackwell forward's bottleneck, and FA4 computes some of them with a
// polynomial on the FMA units).
//
// Method (Cody and Waite's range reduction): x = n + f with n the nearest
// integer and f in [-1/2, 1/2]; 2^f by the polynomial 1 + f*(c1 + f*(c2 +
// f*c3)) in fused multiply-adds; 2^n by adding n to the exponent field.  n
// comes from the rounding of x + 1.5*2^23 (its low mantissa bits then hold n
// in two's complement).  The coefficients minimise the largest relative
// error over [-1/2, 1/2] with the constant term pinned to 1; fit_exp2_poly.py
// beside this file derives them and measures 1.01e-4 in float32.
//
// x is clamped to [-125, 64] first: below, the result stays at 2^-125 (where
// the hardware exponential flushes to 0; either is nothing beside the row's
// largest term, 1, and masked columns are set to 0 after the exponential);
// above, at 2^64, far past the softmax's check that moves its exponent
// reference once a half's sum exceeds 2^16, so no overflow is hidden.  A
// NaN input comes out as 2^-125.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace attn {

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  const float c1 = __uint_as_float(0x3f317afdu);  // 6.932829022e-01
  const float c2 = __uint_as_float(0x3e780627u);  // 2.422109693e-01
  const float c3 = __uint_as_float(0x3d61510cu);  // 5.500893295e-02
  const float2 round_magic = make_float2(12582912.f, 12582912.f);  // 1.5 * 2^23
  x.x = fminf(fmaxf(x.x, -125.f), 64.f);
  x.y = fminf(fmaxf(x.y, -125.f), 64.f);
  const float2 t = fadd2(x, round_magic);      // nearest integer n in the low bits of t
  const float2 f = fsub2(x, fsub2(t, round_magic));
  float2 p = ffma2(make_float2(c3, c3), f, make_float2(c2, c2));
  p = ffma2(p, f, make_float2(c1, c1));
  p = ffma2(p, f, make_float2(1.f, 1.f));
  // 2^n * p: n into the exponent field (p lies in [0.70, 1.42], the result
  // in [2^-126, 2^65): no field overflows)
  const uint32_t ex = __float_as_uint(t.x) << 23, ey = __float_as_uint(t.y) << 23;
  return make_float2(__uint_as_float(__float_as_uint(p.x) + ex), __uint_as_float(__float_as_uint(p.y) + ey));
}

}  // namespace attn
