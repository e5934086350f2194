// Host builder of the dynamic-tree maps, thresholds and the bucket entries.
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

int count_le(const float* t, float v) {
  int c = 0;
  while (c < kCodes - 1 && t[c] <= v) ++c;
  return c;
}

uint32_t to_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return u;
}

// Entry of one bucket of one sign whose values run from v_lo to v_hi
// (v_lo <= v_hi).  `shift` and `low_mask` split a pattern into bucket and
// low bits; negative buckets complement the low bits.  Fails if the bucket
// holds two thresholds, or a threshold outside its pattern range (possible
// only in a clamped first bucket).
int make_entry(const float* t, float v_lo, float v_hi, uint32_t shift, uint32_t low_mask, bool negative,
               uint32_t* out, char* err, size_t errlen) {
  const int c = count_le(t, v_lo);
  uint32_t tl = 1u << kSgnShift;  // no threshold: above every low value of either map
  if (c < kCodes - 1 && t[c] <= v_hi) {
    if (c + 1 < kCodes - 1 && t[c + 1] <= v_hi) {
      std::snprintf(err, errlen, "bucket [%a, %a] holds two thresholds", v_lo, v_hi);
      return -1;
    }
    const uint32_t tb = to_bits(t[c]);
    if ((tb >> shift) != (to_bits(negative ? v_lo : v_hi) >> shift)) {
      std::snprintf(err, errlen, "threshold %a lies outside the patterns of bucket [%a, %a]", t[c], v_lo, v_hi);
      return -1;
    }
    tl = negative ? ((tb & low_mask) ^ low_mask) : (tb & low_mask);
  }
  *out = (static_cast<uint32_t>(c) << kEntShift) + (1u << kEntShift) - tl;
  return 0;
}

int build_entries(const float* ts, const float* tu, uint32_t* ent, char* err, size_t errlen) {
  for (int i = 0; i < kEntries; ++i) ent[i] = 255u << kEntShift;  // padding, never read
  // each stored word is the bucket's E less its lookup word's top bits
  // (tables.h), so that entry + lookup word = E + low bits
  for (uint32_t h = kSgnLo; h <= kSgnHi; ++h) {
    // the first bucket of each sign also takes every smaller magnitude
    // (down to +0.0, and down to the smallest negative subnormal: -0.0 is
    // handed to the lookup as +0.0)
    const float top = from_bits((h << kSgnShift) | kSgnLowMask);
    const float pos_lo = h == kSgnLo ? 0.0f : from_bits(h << kSgnShift);
    const float neg_hi = h == kSgnLo ? -from_bits(1u) : -from_bits(h << kSgnShift);
    const uint32_t jn = h ^ kSgnIdxFlip;  // index of the negative bucket
    uint32_t ep, en;
    if (make_entry(ts, pos_lo, top, kSgnShift, kSgnLowMask, false, &ep, err, errlen) != 0 ||
        make_entry(ts, -top, neg_hi, kSgnShift, kSgnLowMask, true, &en, err, errlen) != 0)
      return -1;
    ent[h - kSgnBase] = ep - (h << kSgnShift);
    ent[jn - kSgnBase] = en - (jn << kSgnShift);
  }
  for (uint32_t h = kUnsLo; h <= kUnsHi; ++h) {
    const float lo = h == kUnsLo ? 0.0f : from_bits(h << kUnsShift);
    uint32_t e;
    if (make_entry(tu, lo, from_bits((h << kUnsShift) | kUnsLowMask), kUnsShift, kUnsLowMask, false, &e, err,
                   errlen) != 0)
      return -1;
    ent[kUnsOff + h - kUnsLo] = e - (h << kUnsShift);
  }
  // Unsigned quantization divides by the block absmax without a
  // tiny-quotient check (exact_div.cuh, unscaled form), so a quotient below
  // 2^-63 may come out with either sign; the lookup clamps it into the first
  // bucket.  That gives code 0, the code of every such quotient, only while
  // the first bucket holds no threshold.
  if (ent[kUnsOff] + (kUnsLo << kUnsShift) != (1u << kEntShift) - (1u << kSgnShift)) {
    std::snprintf(err, errlen, "the first unsigned bucket holds a threshold");
    return -1;
  }
  return 0;
}

}  // namespace

int build_tables(Tables* tab, char* err, size_t errlen) {
  float thr[2][kCodes];
  for (int k = 0; k < 2; ++k) {
    build_map(k == 0, tab->map[k]);
    build_thresholds(tab->map[k], thr[k]);
  }
  return build_entries(thr[0], thr[1], tab->ent, err, errlen);
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
