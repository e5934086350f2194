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
//   entries.  Per bucket E = c * 2^24 + (2^24 - tl), with tl the
//   (complemented, for negative buckets) low bits of the bucket's threshold,
//   or 2^17 when the bucket has none.  For any low < 2^17,
//       code(q) = (E + low(q)) >> 24,  the top byte of the sum,
//   because 2^24 - tl + low lies in [2^24 - 2^17, 2^24 + 2^17) and reaches
//   2^24 exactly when low >= tl.  The sum stays below 2^32: a bucket with
//   c = 255 has no threshold left (E = 2^32 - 2^17), and for c <= 254
//   E <= 255 * 2^24.
//
//   lookup word.  The kernels look up a word x whose top bits are the
//   bucket's table index j and whose low bits are low(q), and the table
//   stores E - j * 2^shift (mod 2^32), so that one add, ent[j] + x, gives
//   E + low(q) with no masking.  The kernels keep the sums and pack the top
//   bytes of four of them into one word of codes with byte permutes.
//
//   Signed map (first moment): bucket h = |pattern| >> 17 (64 per binade:
//   the signed thresholds are at least 1.4% apart), clamped to
//   [kSgnLo, kSgnHi]: magnitudes from 2^-21 (below the smallest nonzero
//   threshold, 5e-7) to 1.016.  With m the pattern of the clamped magnitude
//   and s the sign mask of q (all ones when q is negative),
//       x = m ^ (s & kSgnFlip):
//   m itself for q >= 0; for q < 0 the low bits complemented and bits 11
//   and 0 of the bucket flipped.  Every bucket in [kSgnLo, kSgnHi] has bit
//   11 set, so the negative buckets sit below the positive ones, at
//   (h ^ 1) - 2^11, and the table spans [kSgnLo - 2^11, kSgnHi] from entry 0
//   (the indices between the two ranges are never read).  Bit 0 swaps
//   neighbouring buckets so that the two entries of one magnitude lie
//   2^11 +- 1 words apart, in different shared-memory banks: 2^11 apart
//   they share a bank, and a warp holding both signs of one magnitude (a
//   first moment's usual state) reads them one after the other (per 7B
//   step with bf16 parameters 12.65 against 12.83 ms, with fp32 ones 13.97
//   against 14.12).  Every magnitude below 2^-21
//   shares the first bucket of its sign; that is exact for all of them but
//   -0.0, whose code (that of +0.0, 128) the kernels obtain by adding +0.0
//   to a zero quotient first.
//   Unsigned map (second moment): bucket = pattern >> 16 (128 per binade:
//   its thresholds are 0.7% apart near 1), clamped to [kUnsLo, kUnsHi]
//   (2^-25, below the smallest threshold 5e-8, to 1.008), x = the clamped
//   pattern, entries from kUnsOff on.
//   Lookups clamp only from below (with fmaxf, which also sends NaN to the
//   first bucket): a normalised value is a block's own quotient, in [-1, 1]
//   or NaN (see code_word_signed in kernels.cu), so the bucket of 1.0 is the
//   top one.  A clamped value takes the low bits of the clamp, 0 (or all
//   ones, negative), in a first bucket, which holds no threshold.
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
constexpr uint32_t kSgnNegBit = 0x800u;             // moves negative buckets below the positive ones
constexpr uint32_t kSgnIdxFlip = kSgnNegBit | 1u;   // bucket bits flipped for q < 0
constexpr uint32_t kSgnFlip = (kSgnIdxFlip << kSgnShift) | kSgnLowMask;
constexpr uint32_t kSgnBase = kSgnLo - kSgnNegBit;  // index of entry 0 (lowest negative bucket)
constexpr uint32_t kSgnSpan = kSgnHi - kSgnBase + 1u;
static_assert((kSgnLo & ~(kSgnNegBit - 1u)) == (kSgnHi & ~(kSgnNegBit - 1u)) && (kSgnLo & kSgnNegBit),
              "every signed bucket has bit 11 set");
static_assert(kSgnLo % 2u == 0u && ((kSgnHi ^ 1u) - kSgnNegBit) < kSgnLo,
              "negative indices start at kSgnBase and end below the positive ones");
constexpr uint32_t kUnsShift = 16;                 // unsigned bucket = pattern >> 16
constexpr uint32_t kUnsLowMask = (1u << kUnsShift) - 1u;
constexpr uint32_t kUnsLo = 0x3300u;               // pattern >> 16 of 2^-25
constexpr uint32_t kUnsHi = 0x3F80u;               // pattern >> 16 of 1.0
constexpr uint32_t kUnsOff = kSgnSpan;             // where the unsigned entries start
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
