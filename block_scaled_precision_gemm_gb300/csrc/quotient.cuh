// x / s in binary32, correctly rounded (round to nearest even), for a divisor
// s that a whole block of elements shares: the quantizers' q = x / s.
//
// Method: Markstein's final correction step (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; proof outline in Cornea-Hasegan, Golliver and Markstein,
// "Correctness proofs outline for Newton-Raphson based floating-point divide
// and square root algorithms", ARITH-14, 1999).  If y is the correctly rounded
// reciprocal RN(1/s) and q lies within one ulp of x/s, the remainder
// r = x - q s is exactly representable (one fused multiply-add computes it
// exactly) and RN(q + r y) = RN(x/s).
//
// Here y is computed once per block by one IEEE division.  The estimate
// q0 = RN(x y) lies within 1.5 ulp of x/s; one correction step brings it
// within one ulp (its remainder may round, which only perturbs the
// correction by a relative 2^-23), and a second step, whose remainder is
// exact, gives the correctly rounded quotient.  Five FP32 operations per
// element instead of a division.
//
// Range: the theorem assumes nothing underflows.  block_recip() returns 0
// unless 2^-80 <= s <= 2^126 (the callers then divide); in that range the
// result is RN(x/s) bit for bit whenever neither |x| nor |x/s| is below
// 2^-100.  Otherwise both it and RN(x/s) are below 2^-19 in magnitude with
// x's sign (|x| < 2^-100 gives |x/s| < 2^-20), which every code format here
// (E4M3, E5M2, E2M1, INT8) turns into the same zero code.
// bsmm_selftest_quotient() checks this against the hardware division.
#pragma once

#include <cstdint>

namespace bsmm {

// RN(1/s) for a block's divisor, or 0 outside the range above.
__device__ __forceinline__ float block_recip(float s) {
  return (s >= 0x1p-80f && s <= 0x1p126f) ? __fdiv_rn(1.f, s) : 0.f;
}

__device__ __forceinline__ float with_sign_of(float q, float x) {
  return __uint_as_float((__float_as_uint(q) & 0x7FFFFFFFu) | (__float_as_uint(x) & 0x80000000u));
}

// RN(x / s), given y = block_recip(s) != 0.
__device__ __forceinline__ float quot_rn(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, x), y, q0);
  const float q2 = __fmaf_rn(__fmaf_rn(-q1, s, x), y, q1);
  return with_sign_of(q2, x);
}

// Two quotients by the same s on the packed FP32 pipe, with the sign of a
// zero or tiny quotient left as it falls: for integer codes, which round
// those to 0 either way.
__device__ __forceinline__ float2 quot2_rn_int(float2 x, float s, float y) {
  const float2 ns = make_float2(-s, -s), y2 = make_float2(y, y);
  const float2 q0 = __fmul2_rn(x, y2);
  const float2 q1 = __ffma2_rn(__ffma2_rn(q0, ns, x), y2, q0);
  return __ffma2_rn(__ffma2_rn(q1, ns, x), y2, q1);
}

// Two quotients by the same s, each RN(x / s) with x's sign.
__device__ __forceinline__ float2 quot2_rn(float2 x, float s, float y) {
  const float2 q = quot2_rn_int(x, s, y);
  return make_float2(with_sign_of(q.x, x.x), with_sign_of(q.y, x.y));
}

}  // namespace bsmm
