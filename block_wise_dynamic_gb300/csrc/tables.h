// Code tables shared by the host builder (codebook.cpp) and the kernels.
//
// A quantization code is the index of the nearest entry of a 256-entry
// ascending map ("8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION", section 二 /
// 动态量化).  It equals the number of decision thresholds t[i] (midpoints of
// neighbouring entries) that are <= the normalised value.  Besides the map
// and the thresholds the kernels use one more table to find that count
// without a search:
//
//   bucket table.  For y >= +0 the binary32 bit pattern is monotone in y.
//   Bucket b holds every y whose pattern >> kBktShift equals kBktBase + b
//   (bucket 0 also takes everything below; the last one the values from
//   1.0 up).  bkt[b] = number of thresholds <= the smallest y of the bucket.
//   The builder checks that a bucket contains at most one further threshold,
//   so  count(y) = bkt[b] + (thr[bkt[b]] <= y)  exactly.
#pragma once

#include <cstddef>
#include <cstdint>

namespace bwd {

constexpr int kCodes = 256;
constexpr int kBktShift = 16;                    // 7 mantissa bits per bucket
constexpr int kBktBase = (127 - 26) << 7;        // pattern of 2^-26, >> 16
constexpr int kNumBkt = (127 << 7) - kBktBase + 1;  // through the bucket of 1.0
constexpr int kBktPad = 3344;                    // kNumBkt rounded up to 16

static_assert(kBktPad >= kNumBkt && kBktPad % 16 == 0, "bucket padding");

// Index 0: signed map (first moment), 1: unsigned map (second moment).
struct Tables {
  float map[2][kCodes];   // ascending values
  float thr[2][kCodes];   // 255 thresholds, [255] = +inf
  uint8_t bkt[2][kBktPad];
};

static_assert(sizeof(Tables) % 16 == 0, "tables are copied as 16-byte words");

// Fills *t.  Returns 0, or -1 with a message in err when a table invariant
// fails (which would mean the bucket width is too coarse for the map).
int build_tables(Tables* t, char* err, size_t errlen);

}  // namespace bwd
