// Host builder of the dynamic-tree maps, thresholds and the count table.
//
// "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION", section 二 / 动态量化: an
// 8-bit dynamic tree number is a sign bit, an exponent counted as leading
// zero bits, an indicator bit and a linear fraction; the unsigned variant
// used for the second moment spends the sign bit on the fraction.
//
// With a tail of w bits (7 signed, 8 unsigned), E leading zeros leave
// k = w - 1 - E fraction bits j.  The magnitude uses a decimal exponent and a
// linear grid whose right end point is 1 in every decade:
//     |v| = 10^-E * (0.1 + 0.9 (j + 1) / 2^k) = (2^k + 9 (j + 1)) / (2^k 10^(E+1)).
// Numerator (<= 1280) and denominator (<= 10^8 = 2^8 * 390625) are exact in
// binary32, so one IEEE division gives the binary32 value nearest to the
// exact rational.  Codes are indices into the ascending list of the 256
// values; the signed list holds -0.0 before +0.0 for the two zero patterns.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <limits>

#include "bwd.h"
#include "tables.h"

namespace bwd {
namespace {

float pow10_exact(int e) {
  float r = 1.0f;
  for (int i = 0; i < e; ++i) r *= 10.0f;  // exact up to 10^10
  return r;
}

// Positive magnitudes in ascending order; returns how many (2^w - 1).
int positive_magnitudes(int w, float* out) {
  int c = 0;
  for (int E = w - 1; E >= 0; --E) {  // larger E = smaller decade
    const int k = w - 1 - E;
    const float two_k = static_cast<float>(1 << k);
    const float den = two_k * pow10_exact(E + 1);
    for (int j = 0; j < (1 << k); ++j) {
      const float num = two_k + 9.0f * static_cast<float>(j + 1);
      out[c++] = num / den;
    }
  }
  return c;
}

void build_map(bool is_signed, float* m) {
  float pos[255];
  if (is_signed) {
    const int np = positive_magnitudes(7, pos);  // 127
    for (int i = 0; i < np; ++i) m[i] = -pos[np - 1 - i];
    m[np] = -0.0f;
    m[np + 1] = 0.0f;
    for (int i = 0; i < np; ++i) m[np + 2 + i] = pos[i];
  } else {
    const int np = positive_magnitudes(8, pos);  // 255
    m[0] = 0.0f;
    for (int i = 0; i < np; ++i) m[1 + i] = pos[i];
  }
}

// Threshold i: binary32 nearest to (m[i] + m[i+1]) / 2.  Neighbouring entries
// differ by at most a factor 6, so their sum is exact in binary64; halving is
// exact and the conversion rounds to nearest, ties to even.
void build_thresholds(const float* m, float* t) {
  for (int i = 0; i < kCodes - 1; ++i) {
    const double mid = (static_cast<double>(m[i]) + static_cast<double>(m[i + 1])) * 0.5;
    t[i] = static_cast<float>(mid);
  }
  t[kCodes - 1] = std::numeric_limits<float>::infinity();
}

float from_bits(uint32_t u) {
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// One bucket: values from v_lo to v_hi (v_lo <= v_hi).  Stores the count of
// thresholds <= v_lo and checks that (v_lo, v_hi] holds at most one more.
int fill_bucket(const float* t, float v_lo, float v_hi, uint8_t* out, char* err, size_t errlen) {
  int c = 0;
  while (c < kCodes - 1 && t[c] <= v_lo) ++c;
  *out = static_cast<uint8_t>(c);
  if (c + 1 < kCodes - 1 && !(t[c + 1] > v_hi)) {
    std::snprintf(err, errlen, "bucket [%a, %a] holds two thresholds", v_lo, v_hi);
    return -1;
  }
  return 0;
}

int build_counts(const float* ts, const float* tu, uint8_t* cnt, char* err, size_t errlen) {
  std::memset(cnt, 255, kCntPad);  // buckets no normalised value reaches
  const uint32_t sh = kCntSignedShift, low = (1u << kCntSignedShift) - 1u;
  for (uint32_t i = 0; i <= (kCntSignedMax & 0x1fffu); ++i) {
    // non-negative patterns: the lowest value has the smallest pattern
    if (fill_bucket(ts, from_bits(i << sh), from_bits((i << sh) | low), &cnt[i], err, errlen) != 0) return -1;
    // negative patterns: the lowest value has the largest pattern
    const uint32_t n = i | 0x4000u;
    if (fill_bucket(ts, from_bits((n << sh) | low), from_bits(n << sh), &cnt[n], err, errlen) != 0) return -1;
  }
  for (uint32_t h = kCntUnsignedLo; h <= kCntUnsignedHi; ++h) {
    // the first bucket also takes every value below 2^-26
    const float lo = h == kCntUnsignedLo ? 0.0f : from_bits(h << 16);
    if (fill_bucket(tu, lo, from_bits((h << 16) | 0xffffu), &cnt[kCntUnsignedOff + h - kCntUnsignedLo], err,
                    errlen) != 0)
      return -1;
  }
  return 0;
}

}  // namespace

int build_tables(Tables* tab, char* err, size_t errlen) {
  for (int k = 0; k < 2; ++k) {
    build_map(k == 0, tab->map[k]);
    build_thresholds(tab->map[k], tab->thr[k]);
  }
  return build_counts(tab->thr[0], tab->thr[1], tab->cnt, err, errlen);
}

}  // namespace bwd

extern "C" bwd_status bwd_build_map(bwd_map_kind kind, float* map_out, float* thresholds_out) {
  if (kind != BWD_MAP_SIGNED && kind != BWD_MAP_UNSIGNED) return BWD_ERR_INVALID_ARG;
  float m[bwd::kCodes];
  float t[bwd::kCodes];
  bwd::build_map(kind == BWD_MAP_SIGNED, m);
  bwd::build_thresholds(m, t);
  if (map_out) std::memcpy(map_out, m, sizeof m);
  if (thresholds_out) std::memcpy(thresholds_out, t, sizeof(float) * (bwd::kCodes - 1));
  return BWD_OK;
}

extern "C" int64_t bwd_num_blocks(int64_t n) {
  if (n < 0) return -1;
  return (n + BWD_BLOCK - 1) / BWD_BLOCK;
}
