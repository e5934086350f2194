// Code tables shared by the host builder (codebook.cpp) and the kernels.
//
// A quantization code is the index of the nearest entry of a 256-entry
// ascending map ("8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION", section 二 /
// 动态量化).  It equals the number of decision thresholds t[i] (midpoints of
// neighbouring entries) that are <= the normalised value q.  Besides the maps
// and the thresholds the kernels use one more table to find that count
// without a search:
//
//   count table.  Binary32 values whose bit patterns agree in the top 16 bits
//   form a bucket (7 mantissa bits: 128 buckets per binade).  For a bucket
//   with lowest value v_lo (the most negative one for negative patterns),
//   cnt[bucket] = number of thresholds <= v_lo.  The builder checks that no
//   bucket holds more than one further threshold, so for any q in the bucket
//       code(q) = cnt[bucket] + (thr[cnt[bucket]] <= q)
//   exactly, ties and signed zeros included.  Signed map: bucket = pattern
//   >> 16, covering [-1.0078, 1.0078) in [0, 0xBF80].  Unsigned map: bucket =
//   (pattern >> 16) + 0x4000, placed in the gap [0x3F81, 0x7FFF] the signed
//   map never uses (its positive patterns stop at 0x3F80).
#pragma once

#include <cstddef>
#include <cstdint>

namespace bwd {

constexpr int kCodes = 256;
constexpr uint32_t kCntSignedMax = 0xBF80u;    // bucket of -1.0 (clamp for signed lookups)
constexpr uint32_t kCntUnsignedMax = 0x3F80u;  // bucket of +1.0 (clamp for unsigned lookups)
constexpr uint32_t kCntUnsignedOff = 0x4000u;  // where the unsigned buckets start
constexpr int kCntPad = 49040;                 // 0xBF81 entries rounded up to 16

static_assert(kCntPad >= static_cast<int>(kCntSignedMax) + 1, "count table size");
static_assert(kCntUnsignedOff + kCntUnsignedMax < 0x8000u, "unsigned buckets fit the gap");

// Index 0: signed map (first moment), 1: unsigned map (second moment).
struct Tables {
  float map[2][kCodes];   // ascending values
  float thr[2][kCodes];   // 255 thresholds, [255] = +inf
  uint8_t cnt[kCntPad];   // count table, both maps
};

static_assert(sizeof(Tables) % 16 == 0, "tables are copied as 16-byte words");

// Fills *t.  Returns 0, or -1 with a message in err when a table invariant
// fails (which would mean the bucket width is too coarse for the map).
int build_tables(Tables* t, char* err, size_t errlen);

}  // namespace bwd
