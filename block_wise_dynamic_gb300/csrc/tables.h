// Code tables shared by the host builder (codebook.cpp) and the kernels.
//
// A quantization code is the index of the nearest entry of a 256-entry
// ascending map ("8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION", section 二 /
// 动态量化).  It equals the number of decision thresholds t[i] (midpoints of
// neighbouring entries) that are <= the normalised value q.  The kernels find
// that count with one table read and no search:
//
//   buckets.  Binary32 values of one sign whose bit patterns agree in their
//   top bits form a bucket.  The builder checks that every bucket holds at
//   most one threshold, so inside a bucket the count is c (the thresholds
//   below the bucket) or c + 1 (q at or above the bucket's threshold).
//   Inside a bucket of positive values, q >= t exactly when the low pattern
//   bits of q are >= those of t; for negative values the order of the low
//   bits is reversed, so they are complemented first ("low" below).
//
//   entries.  One 32-bit word per bucket, E = c * 2^24 + (2^24 - tl), with tl
//   the (complemented, for negative buckets) low bits of the bucket's
//   threshold, or 2^17 when the bucket has none.  For any low < 2^17,
//       code(q) = (E + low(q)) >> 24,  the top byte of the sum,
//   because 2^24 - tl + low lies in [2^24 - 2^17, 2^24 + 2^17) and reaches
//   2^24 exactly when low >= tl.  The sum stays below 2^32: a bucket with
//   c = 255 has no threshold left (E = 2^32 - 2^17), and for c <= 254
//   E <= 255 * 2^24.  The kernels keep the sums and pack the top bytes of
//   four of them into one word of codes with byte permutes.
//
//   Signed map (first moment): bucket = |pattern| >> 17 (64 per binade: the
//   signed thresholds are at least 1.4% apart), clamped to [kSgnLo, kSgnHi]:
//   magnitudes from 2^-21 (below the smallest nonzero threshold, 5e-7) to
//   1.016.  Entries [0, kSgnN) are the positive buckets, [kSgnN, 2 kSgnN) the
//   negative ones.  Every magnitude below 2^-21 shares the first bucket of its
//   sign; that is exact for all of them but -0.0, whose code (that of +0.0,
//   128) the kernels obtain by adding +0.0 to a zero quotient first.
//   Unsigned map (second moment): bucket = pattern >> 16 (128 per binade: its
//   thresholds are 0.7% apart near 1), clamped to [kUnsLo, kUnsHi] (2^-25,
//   below the smallest threshold 5e-8, to 1.008), from kUnsOff on.
//   Lookups clamp only from below (with fmaxf, which also sends NaN to the
//   first bucket): a normalised value is a block's own quotient, in [-1, 1]
//   or NaN (see code_word_signed in kernels.cu), so the bucket of 1.0 is the
//   top one.
#pragma once

#include <cstddef>
#include <cstdint>

namespace bwd {

constexpr int kCodes = 256;
constexpr uint32_t kEntShift = 24;                 // code = (entry + low) >> kEntShift
constexpr uint32_t kSgnShift = 17;                 // signed bucket = |pattern| >> 17
constexpr uint32_t kSgnLowMask = (1u << kSgnShift) - 1u;
constexpr uint32_t kSgnLo = 0x1A80u;               // bucket of 2^-21
constexpr uint32_t kSgnHi = 0x1FC0u;               // bucket of 1.0
constexpr uint32_t kSgnN = kSgnHi - kSgnLo + 1u;   // buckets per sign
constexpr uint32_t kUnsShift = 16;                 // unsigned bucket = pattern >> 16
constexpr uint32_t kUnsLowMask = (1u << kUnsShift) - 1u;
constexpr uint32_t kUnsLo = 0x3300u;               // pattern >> 16 of 2^-25
constexpr uint32_t kUnsHi = 0x3F80u;               // pattern >> 16 of 1.0
constexpr uint32_t kUnsOff = 2u * kSgnN;           // where the unsigned entries start
constexpr int kEntries = static_cast<int>((kUnsOff + kUnsHi - kUnsLo + 1u + 3u) / 4u * 4u);

// Index 0: signed map (first moment), 1: unsigned map (second moment).
struct Tables {
  float map[2][kCodes];    // ascending values
  uint32_t ent[kEntries];  // bucket entries, both maps
};

static_assert(sizeof(Tables) % 16 == 0, "tables are copied as 16-byte words");

// Fills *t.  Returns 0, or -1 with a message in err when a table invariant
// fails (which would mean the bucket width is too coarse for the map).
int build_tables(Tables* t, char* err, size_t errlen);

}  // namespace bwd
