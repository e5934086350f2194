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
//
// Unscaled form (div_unscaled2).  When the divisor's biased exponent lies in
// [89, 252], that is 2^-38 <= a < 2^126, the scaling can be left out: Y =
// RN(1 / a) equals y 2^k exactly and is normal, and q0 = RN(x Y), r = x - a q0
// (one fma), RN(q0 + r Y) take the same values as the scaled sequence times
// powers of two, so the result is RN(x / a) as long as r is exact.  r is a
// multiple of 2^(e_a + e_q0 - 46) (e_ the unbiased exponents of a and q0)
// below 2^(e_a + e_q0 - 22) in magnitude, so it is representable, subnormal
// or not, whenever e_a + e_q0 >= -103, which |x / a| >= 2^-64 guarantees.
// Below 2^-64 the unscaled result stays within 2^-22 |x / a| + 2^-111 of x / a
// (r is then off by at most half a subnormal step, times Y <= 2^38), so its
// magnitude is below 2^-63, but its sign may differ from that of x.  This
// saves one multiply per dividend.
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

// Packed binary32 pairs (PTX .f32x2, sm_100 and later): each lane of the
// pair is one IEEE round-to-nearest operation, exactly as the scalar one,
// at half the issue cost.  Measured: a packed multiply whose result feeds a
// packed add can come out contracted into one fused multiply-add despite
// the .rn qualifier, so sums of products that must round twice (the Adam
// moments) add in scalar __fadd_rn (their products may be packed); packed
// adds are used only where no multiply feeds them (the exact division,
// whose products feed fused operations by design, and the approximate
// parameter update).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }

__device__ __forceinline__ float div_fast(const Divisor& d, float x) {
  const float xs = __fmul_rn(x, d.scale);
  const float q0 = __fmul_rn(xs, d.y);
  const float r = __fmaf_rn(-d.a, q0, xs);
  return __fmaf_rn(r, d.y, q0);
}

// The same for two dividends at once with packed operations: per lane the
// identical sequence of IEEE operations (no multiply here feeds an add).
__device__ __forceinline__ float2 div_fast2(const Divisor& d, float2 x) {
  const float2 xs = mul2(x, dup2(d.scale));
  const float2 q0 = mul2(xs, dup2(d.y));
  const float2 r = fma2(dup2(-d.a), q0, xs);
  return fma2(r, dup2(d.y), q0);
}

// Divisors for which div_unscaled2 is exact on quotients of magnitude
// >= 2^-64 (see the header comment): positive, exponent field in [89, 252],
// one unsigned compare.  Their reciprocal Y = RN(1 / a) (__frcp_rn) is
// normal.
__device__ __forceinline__ bool unscaled_ok(float a) {
  return __float_as_uint(a) - (89u << 23) < ((253u - 89u) << 23);
}

__device__ __forceinline__ float div_unscaled(float x, float a, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-a, q0, x);
  return __fmaf_rn(r, y, q0);
}

__device__ __forceinline__ float2 div_unscaled2(float2 x, float a, float y) {
  const float2 y2 = dup2(y);
  const float2 q0 = mul2(x, y2);
  const float2 r = fma2(dup2(-a), q0, x);
  return fma2(r, y2, q0);
}

}  // namespace bwd
