// Exhaustive check of the library's bucket entries (csrc/tables.h): for every
// binary32 pattern q with |q| <= 1 the one-read lookup the kernels perform
// must give the number of thresholds <= q, and no pattern the kernels can
// look up (|q| <= 1 or NaN: a block's own quotients) may index outside the
// table.
//
// The thresholds come from the file named by argv[1] (255 signed, then 255
// unsigned binary32 values, written by the test from the CPU oracle); the
// entries come from the library's own builder.  The two lookups below
// restate code_word_signed / code_word_unsigned_nonneg of csrc/kernels.cu (whose
// top byte is the code) on the host:
// the kernels hand -0.0 to the signed lookup as +0.0, and so does this check.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <thread>
#include <vector>

#include "tables.h"

namespace {

const bwd::Tables* g_tab;
float g_ts[255], g_tu[255];

float fbits(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

uint32_t lookup_signed(float q, bool* oob) {
  const uint32_t m = bits(std::fmax(std::fabs(q), fbits(bwd::kSgnLo << bwd::kSgnShift)));
  const uint32_t s = static_cast<uint32_t>(static_cast<int32_t>(bits(q)) >> 31);
  const uint32_t x = m ^ (s & bwd::kSgnFlip);
  const uint32_t i = (x >> bwd::kSgnShift) - bwd::kSgnBase;
  if (i >= bwd::kSgnSpan) { *oob = true; return 0; }
  return (g_tab->ent[i] + x) >> bwd::kEntShift;
}

uint32_t lookup_unsigned(float q, bool* oob) {
  const uint32_t x = bits(std::fmax(q, fbits(bwd::kUnsLo << bwd::kUnsShift)));
  const uint32_t i = bwd::kUnsOff - bwd::kUnsLo + (x >> bwd::kUnsShift);
  if (i < bwd::kUnsOff || i >= static_cast<uint32_t>(bwd::kEntries)) { *oob = true; return 0; }
  return (g_tab->ent[i] + x) >> bwd::kEntShift;
}

uint32_t count_le(const float* t, float q) {  // thresholds ascending
  uint32_t lo = 0, hi = 255;
  while (lo < hi) {
    const uint32_t m = (lo + hi) / 2;
    if (t[m] <= q) lo = m + 1; else hi = m;
  }
  return lo;
}

}  // namespace

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  FILE* f = std::fopen(argv[1], "rb");
  if (!f || std::fread(g_ts, 4, 255, f) != 255 || std::fread(g_tu, 4, 255, f) != 255) return 2;
  std::fclose(f);
  static bwd::Tables tab;
  char err[256] = {0};
  if (bwd::build_tables(&tab, err, sizeof err) != 0) { std::printf("build failed: %s\n", err); return 1; }
  g_tab = &tab;

  unsigned nt = std::thread::hardware_concurrency();
  nt = nt < 1 ? 1 : (nt > 32 ? 32 : nt);
  std::atomic<long> checked{0}, bad{0}, oob{0};
  std::vector<std::thread> pool;
  for (unsigned w = 0; w < nt; ++w) {
    pool.emplace_back([&, w] {
      long c = 0, b = 0, o = 0;
      const uint64_t lo = (0x100000000ull * w) / nt, hi = (0x100000000ull * (w + 1)) / nt;
      for (uint64_t u = lo; u < hi; ++u) {
        const uint32_t pb = static_cast<uint32_t>(u);
        const float q = fbits(pb);
        if (!std::isnan(q) && std::fabs(q) > 1.0f) continue;  // never looked up
        // quotients come out of arithmetic, whose NaNs are quiet: signaling
        // NaN patterns are never looked up either
        if (std::isnan(q) && !(pb & 0x00400000u)) continue;
        bool x = false;
        const uint32_t cs = lookup_signed(q == 0.0f ? 0.0f : q, &x);
        const uint32_t cu = lookup_unsigned(q, &x);
        if (x) { ++o; continue; }
        if (std::isnan(q)) continue;
        ++c;
        if (cs != count_le(g_ts, q)) { if (b++ < 5) std::printf("signed %08x: %u vs %u\n", pb, cs, count_le(g_ts, q)); }
        if (!(pb >> 31)) {
          ++c;
          if (cu != count_le(g_tu, q)) { if (b++ < 5) std::printf("unsigned %08x: %u vs %u\n", pb, cu, count_le(g_tu, q)); }
        }
      }
      checked += c; bad += b; oob += o;
    });
  }
  for (auto& t : pool) t.join();
  std::printf("checked %ld mismatches %ld out_of_bounds %ld threads %u\n", checked.load(), bad.load(), oob.load(), nt);
  return (bad.load() || oob.load() || checked.load() != 3196059651L) ? 1 : 0;
}
