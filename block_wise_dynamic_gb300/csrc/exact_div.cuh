// Division of many dividends by one divisor, rounded to nearest exactly like
// the IEEE binary32 quotient x / a, without a full division per element.
//
// Method (Markstein's correction step, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; also
// Muller et al., "Handbook of Floating-Point Arithmetic", the theorem on
// correcting a faithful quotient with a correctly rounded reciprocal):
// with y = RN(1/a), q0 = RN(x y), the remainder r = x - a q0 is exact when
// computed by one fused multiply-add, and RN(q0 + r y) = RN(x / a), as long
// as nothing underflows.  To keep every intermediate in the normal range the
// divisor is first scaled by a power of two into [1, 2) (the dividend by the
// same power, which is exact or underflows only for quotients below 2^-126).
//
// Callers must treat quotients of magnitude below 2^-64 as approximate: the
// result then still has the right sign and is tiny, but it may differ from
// RN(x / a) (for instance -0.0 against a negative subnormal).  The tests
// compare this routine with div.rn over every binary32 significand.
#pragma once

#include <cstdint>

namespace bwd {

struct Divisor {
  float a;      // divisor significand, in [1, 2)
  float y;      // RN(1 / a)
  float scale;  // 2^k such that original divisor * 2^k == a
  bool fast;    // false: divisor zero, subnormal, huge or not finite
};

// Divisors with a biased exponent in [lo_exp, 253] take the fast path; the
// caller picks lo_exp (1 accepts every normal divisor).
__device__ __forceinline__ Divisor make_divisor(float d, uint32_t lo_exp) {
  const uint32_t b = __float_as_uint(d);
  const uint32_t e = (b >> 23) & 0xffu;
  Divisor r;
  r.fast = (b >> 31) == 0u && e >= lo_exp && e <= 253u;
  r.a = __uint_as_float((b & 0x007fffffu) | 0x3f800000u);
  r.scale = __uint_as_float((254u - (r.fast ? e : 127u)) << 23);
  r.y = __frcp_rn(r.a);
  return r;
}

__device__ __forceinline__ float div_fast(const Divisor& d, float x) {
  const float xs = __fmul_rn(x, d.scale);
  const float q0 = __fmul_rn(xs, d.y);
  const float r = __fmaf_rn(-d.a, q0, xs);
  return __fmaf_rn(r, d.y, q0);
}

}  // namespace bwd
