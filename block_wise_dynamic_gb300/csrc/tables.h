// Code tables shared by the host builder (codebook.cpp) and the kernels.
//
// A quantization code is the index of the nearest entry of a 256-entry
// ascending map ("8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION", section 二 /
// 动态量化).  It equals the number of decision thresholds t[i] (midpoints of
// neighbouring entries) that are <= the normalised value q.  Besides the maps
// and the thresholds the kernels use one more table to find that count
// without a search:
//
//   count tables.  Binary32 values whose bit patterns agree in their top bits
//   form a bucket.  For a bucket with lowest value v_lo (the most negative
//   one for negative patterns), cnt[bucket] = number of thresholds <= v_lo.
//   The builder checks that no bucket holds more than one further threshold,
//   so for any q in the bucket
//       code(q) = cnt[bucket] + (thr[cnt[bucket]] <= q)
//   exactly, ties and signed zeros included.
//
//   Signed map (first moment): bucket = pattern >> 17 (64 buckets per binade,
//   fine enough because neighbouring signed thresholds are at least 1.4%
//   apart), [0, 0x1FC0] for [0, 1.016) and [0x4000, 0x5FC0] for (-1.016, -0];
//   lookups clamp the bucket to 0x5FC0.
//   Unsigned map (second moment): bucket = pattern >> 16 (128 per binade:
//   its thresholds are 0.7% apart near 1), clamped to [0x3280, 0x3F80], i.e.
//   values from 2^-26 (below the smallest threshold, 5e-8) to 1.008; stored
//   from kCntUnsignedOff on.
//   Entries no normalised value reaches hold 255.  The tables stay small
//   (27 KB) on purpose: shared memory and the L1 cache share one array per
//   SM, and the fused kernel keeps its global loads in flight in L1.
#pragma once

#include <cstddef>
#include <cstdint>

namespace bwd {

constexpr int kCodes = 256;
constexpr uint32_t kCntSignedShift = 17;
constexpr uint32_t kCntSignedMax = 0x5FC0u;    // bucket of -1.0 (clamp for signed lookups)
constexpr uint32_t kCntUnsignedLo = 0x3280u;   // pattern >> 16 of 2^-26
constexpr uint32_t kCntUnsignedHi = 0x3F80u;   // pattern >> 16 of 1.0
constexpr uint32_t kCntUnsignedOff = 0x5FD0u;  // where the unsigned buckets start
constexpr int kCntPad = 27872;                 // kCntUnsignedOff + 0xD01, rounded up to 16

static_assert(kCntUnsignedOff > kCntSignedMax, "unsigned buckets follow the signed ones");
static_assert(kCntPad >= static_cast<int>(kCntUnsignedOff + kCntUnsignedHi - kCntUnsignedLo + 1), "size");

// Index 0: signed map (first moment), 1: unsigned map (second moment).
struct Tables {
  float map[2][kCodes];   // ascending values
  float thr[2][kCodes];   // 255 thresholds, [255] = +inf
  uint8_t cnt[kCntPad];   // count tables, both maps
};

static_assert(sizeof(Tables) % 16 == 0, "tables are copied as 16-byte words");

// Fills *t.  Returns 0, or -1 with a message in err when a table invariant
// fails (which would mean the bucket width is too coarse for the map).
int build_tables(Tables* t, char* err, size_t errlen);

}  // namespace bwd
