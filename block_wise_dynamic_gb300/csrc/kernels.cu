// sm_103a kernels and the C ABI of the 8-bit block-wise dynamic Adam library.
//
// Method: "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (summary on
// wiki.neutronadmin.com/news/16836).  Section 二 / 逐块量化: blocks of 2048
// elements are normalised by their own absmax, independently of each other;
// section 二 / 动态量化: codes index a dynamic-tree map (signed for the first
// moment, unsigned for the second); section 二, opening paragraph: the
// optimizer dequantizes its states, updates in high precision (fp32) and
// stores them quantized again.
//
// Work decomposition.  A group of 128 threads owns one 2048-element block at a
// time and the groups walk the blocks with a grid stride (grid = SMs x
// resident CTAs).  The fused step runs one CTA per SM, of seven groups with
// fp32 parameters and six with 16-bit ones (the register file divided among
// them: 72 and 80 registers a thread), so the code tables sit in shared
// memory once per SM and leave the rest of the unified array to L1 for the
// loads in flight (three 256-thread CTAs per SM, each with its own copy, ran
// 4% slower); the standalone quantizer runs two CTAs of four groups.  Thread t of a group owns the 16 elements 4 t + 512 k + j (k, j < 4)
// of its block ("quads" of 4 elements, 4 x 128 = 512 elements apart), so
// every warp-wide load or store touches one contiguous span (512 B of fp32,
// 256 B of bf16, 128 B of codes) and is fully coalesced.  The block absmax is
// a warp reduction and a pass over the group's four warps through shared
// memory, synchronised by a named barrier per group.  The maps and the
// bucket entries (tables.h) are copied once per CTA into dynamic shared memory.
// The signed standalone quantizer also stages each group's next block in
// shared memory (cp.async); the dequantizer writes each block's output from
// shared memory with one bulk copy.
//
// Exactness.  Every operation that decides a code is IEEE binary32 with
// explicit round-to-nearest intrinsics (no contracted multiply-add): the
// absmax, the quotient x / absmax (exact_div.cuh gives the correctly rounded
// quotient from a per-block reciprocal; tiny negative quotients, where -0.0
// and a negative subnormal give different codes, fall back to div.rn) and
// the threshold compare (an integer compare of pattern bits inside a bucket,
// the same decision for every binary32 value; tables.h).  The moments use
// the same operations, in the same order, as the CPU oracle; the parameter
// update uses approximate sqrt / rcp (a few ulps of the update term).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <type_traits>

#include "bwd.h"
#include "exact_div.cuh"
#include "host_util.h"
#include "tables.h"

namespace {

using bwd::kCodes;

constexpr int kGroup = 128;                   // threads per 2048-element block
constexpr int kPer = BWD_BLOCK / kGroup;      // 16 elements per thread
constexpr int kQuads = kPer / 4;              // 4-element quads per thread
constexpr int kSpan = 4 * kGroup;             // elements between a thread's quads
constexpr int kGroupWarps = kGroup / 32;      // 4
// Adam: blocks in flight per CTA, one CTA per SM (adam_groups below): seven
// 128-thread groups (896 threads, 72 registers) with fp32 parameters and
// 16-bit gradients, six (768 threads, 80 registers) otherwise.
constexpr int kQGroups = 4;                   // blocks in flight per CTA (quantize)
constexpr int kQCta = kGroup * kQGroups;      // 512 threads
constexpr int kDeqThreads = 256;              // dequantize: 8 elements per thread
constexpr int kMaxTensors = 448;              // per launch, bounded by kernel parameter space
constexpr int kMaxDevices = 64;
constexpr int kTablesBytes = static_cast<int>(sizeof(bwd::Tables));

static_assert(kPer % 4 == 0 && kGroupWarps % 4 == 0, "quads of 4 elements, partials read as float4");

__device__ bwd::Tables g_tables;  // immutable after the first upload per device

// --------------------------------------------------------------------------
// device helpers

// Max over a warp of non-negative values: their bit patterns order like the
// values, so one unsigned integer reduction (redux.sync) does it.  Every
// caller passes magnitudes (|m|, v >= 0, |x|); a NaN, outside the method,
// wins here where fmaxf would drop it, and still indexes nothing out of
// bounds downstream.
__device__ __forceinline__ float warp_max(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// Three-input max (sm_100 and later); the .abs form takes magnitudes.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3abs(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3abs(float a, float b, float c) {
  float d;
  asm("min.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Named barrier of one 128-thread group (barrier 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "n"(kGroup) : "memory");
}

// Element of the block owned by slot j (0..15) of thread t.
__device__ __forceinline__ int slot(int t, int j) { return 4 * t + kSpan * (j >> 2) + (j & 3); }

__device__ __forceinline__ int64_t rem_in_block(int64_t n, int64_t base) {
  const int64_t r = n - base;
  return r < BWD_BLOCK ? r : BWD_BLOCK;
}

__device__ __forceinline__ uint32_t byte_of(uint32_t w, int k) { return (w >> (8 * k)) & 0xffu; }

// The same byte by one byte permute (PRMT), which the fp32-parameter fused
// step uses for its dequantizing lookups.  Against shifts and masks, ms per
// 7B step: bf16 gradients 13.98 against 14.13, fp32 gradients 15.98 against
// 16.90, fp16 gradients 13.59-13.67 against 14.0-14.3.  (The
// 16-bit-parameter step forms its lookup offsets with one permute each too:
// see its lane-private map copies.)
__device__ __forceinline__ uint32_t byte_prmt(uint32_t w, int k) {
  return __byte_perm(w, 0u, 0x4440u | static_cast<uint32_t>(k));
}

__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return a | (b << 8) | (c << 16) | (d << 24);
}

__device__ __forceinline__ void copy_to_smem(void* dst, const void* src, int bytes) {
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = static_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x) d[i] = s[i];
}

// Streaming global loads that bypass L1 allocation (each byte is read
// once): L1 capacity stays free for the requests in flight.
__device__ __forceinline__ float4 ld_stream_f4(const void* p) {
  float4 r;
  asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  uint2 r;
  asm volatile("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_stream_u1(const void* p) {
  uint32_t r;
  asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}



// Hint: bring `bytes` (multiple of 16, 16-byte aligned) of global memory into
// L2.  Nothing waits for it, so it cannot stall or hang anything.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Code word of a normalised value (see the bucket entries in tables.h): one
// table read; the code is the word's top byte.  Signed map, -0.0 passed as
// +0.0.
//
// Range of q.  Every q here is a quotient x / absmax of its own block, and
// the block absmax is at least every finite |x| of the block (the running
// maxima start from +0 and max / fmaxf return the non-NaN operand, so no
// NaN ever reaches them); the quotient is exactly rounded, so |q| <= 1.  A
// NaN or infinite x makes q a (quiet, as every arithmetic NaN) NaN, or +-0
// beside an infinite absmax.  So |q| <= 1 or q is a quiet NaN, and the only
// clamp needed is the lower one, which also sends NaN (fmaxf returns the
// other operand) to the first bucket: every lookup stays in the table.
// The lookup word x carries the table index in its top bits and the low
// bits below them; one logic operation folds the sign into both.
__device__ __forceinline__ uint32_t code_word_signed(float q, const bwd::Tables& tab) {
  const uint32_t m = __float_as_uint(fmaxf(fabsf(q), __uint_as_float(bwd::kSgnLo << bwd::kSgnShift)));
  const uint32_t s = static_cast<uint32_t>(static_cast<int32_t>(__float_as_uint(q)) >> 31);
  const uint32_t x = m ^ (s & bwd::kSgnFlip);
  return tab.ent[(x >> bwd::kSgnShift) - bwd::kSgnBase] + x;
}

// Unsigned map, q in [+0, 1] or NaN (the second moment is never negative;
// same range argument as above).
__device__ __forceinline__ uint32_t code_word_unsigned_nonneg(float q, const bwd::Tables& tab) {
  const uint32_t x = __float_as_uint(fmaxf(q, __uint_as_float(bwd::kUnsLo << bwd::kUnsShift)));
  return tab.ent[bwd::kUnsOff - bwd::kUnsLo + (x >> bwd::kUnsShift)] + x;
}

// Unsigned map, any sign: every threshold is positive, so a negative input
// has code 0 (word 0).
__device__ __forceinline__ uint32_t code_word_unsigned(float q, const bwd::Tables& tab) {
  const uint32_t c = code_word_unsigned_nonneg(q, tab);
  return (__float_as_uint(q) >> 31) ? 0u : c;
}

// Codes of 16 values of one block with absmax a.  The fast path is straight
// line (one exact quotient per value from the block's reciprocal, see
// exact_div.cuh).  Quotients of magnitude below 2^-99 may be off there; only a
// negative one can change a code (-0.0 -> code 128, a negative subnormal ->
// code 127).  Read as signed integers, the bit patterns of -0.0 and of the
// negative values closest to zero are the smallest of all, so one integer
// min over the quotients flags a block that has one (a -0.0 quotient
// included); its values with the sign bit set are then redone with IEEE
// division, and a zero quotient is looked up as +0.0.
//
// An absmax in [2^-38, 2^126) takes the unscaled division instead, exact
// for quotients of magnitude >= 2^-64; smaller ones come out below 2^-63 in
// magnitude with a sign that may be wrong.  For the signed map a
// three-input min of magnitudes flags a block with a quotient below 2^-63,
// and there every value with |RN(x Y)| < 2^-62 (every true quotient below
// 2^-64 among them) is redone with IEEE division.  The unsigned map needs
// no check: all its thresholds lie above 2^-25, a negative quotient has
// code 0 (any-sign lookup), and a non-negative lookup of a value below
// 2^-25, of either sign, reads the first bucket, which holds no threshold
// (checked when the tables are built) and so gives code 0, the code of
// every true quotient there.
template <bool kSigned, bool kAnySign>
__device__ __forceinline__ void quantize_quads(const float (&x)[kPer], float a, const bwd::Tables& tab,
                                               uint32_t (&w)[kQuads]) {
  uint32_t c[kPer];  // code words (code in the top byte)
  if (bwd::unscaled_ok(a)) {
    const float y = __frcp_rn(a);  // RN(1 / a), a normal number for such a
    float mq = 1.0f;               // smallest quotient magnitude (m only)
#pragma unroll
    for (int j = 0; j < kPer; j += 2) {
      const float2 q = bwd::div_unscaled2(make_float2(x[j], x[j + 1]), a, y);
      if (kSigned) mq = min3abs(mq, q.x, q.y);
      c[j] = kSigned ? code_word_signed(q.x, tab) : (kAnySign ? code_word_unsigned(q.x, tab) : code_word_unsigned_nonneg(q.x, tab));
      c[j + 1] = kSigned ? code_word_signed(q.y, tab) : (kAnySign ? code_word_unsigned(q.y, tab) : code_word_unsigned_nonneg(q.y, tab));
    }
    if (kSigned && mq < 0x1p-63f) {
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (fabsf(__fmul_rn(x[j], y)) < 0x1p-62f)
          c[j] = code_word_signed(__fadd_rn(__fdiv_rn(x[j], a), 0.0f), tab);  // -0.0 -> +0.0
    }
  } else if (a == 0.0f) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) c[j] = kSigned ? (128u << 24) : 0u;
  } else {
    const bwd::Divisor d = bwd::make_divisor(a, 1u);
    if (d.fast) {
      int minb = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kPer; j += 2) {
        const float2 q = bwd::div_fast2(d, make_float2(x[j], x[j + 1]));
        if (kSigned) minb = min(minb, min(__float_as_int(q.x), __float_as_int(q.y)));
        c[j] = kSigned ? code_word_signed(q.x, tab) : (kAnySign ? code_word_unsigned(q.x, tab) : code_word_unsigned_nonneg(q.x, tab));
        c[j + 1] = kSigned ? code_word_signed(q.y, tab) : (kAnySign ? code_word_unsigned(q.y, tab) : code_word_unsigned_nonneg(q.y, tab));
      }
      if (kSigned && minb <= static_cast<int>(0x8E000000u)) {
#pragma unroll
        for (int j = 0; j < kPer; ++j)
          if (__float_as_int(x[j]) < 0 && bwd::div_fast(d, x[j]) > -0x1p-99f)
            c[j] = code_word_signed(__fadd_rn(__fdiv_rn(x[j], a), 0.0f), tab);  // -0.0 -> +0.0
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const float q = __fdiv_rn(x[j], a);
        c[j] = kSigned ? code_word_signed(__fadd_rn(q, 0.0f), tab) : code_word_unsigned(q, tab);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kQuads; ++k)
    w[k] = __byte_perm(__byte_perm(c[4 * k], c[4 * k + 1], 0x0073), __byte_perm(c[4 * k + 2], c[4 * k + 3], 0x0073), 0x5410);
}

// Max over the 128 threads of a group of non-negative values; every thread
// gets the result.
// `red` is this group's [2 parities][values][4 warps] scratch.  With
// kAllLanes every lane stores its warp's (equal) maximum, which needs no
// branch: the 16-bit-parameter fused step 11.18 against 11.36 ms per 7B
// step; the fp32-parameter one (13.93 against 13.62) and the signed
// quantizer (207 against 196 us) run faster with lane 0 alone.
template <int kVals, bool kAllLanes = false>
__device__ __forceinline__ void group_max(float (&v)[kVals], float* red, int parity, int group, int t) {
  const int lane = t & 31, warp = t >> 5;
#pragma unroll
  for (int i = 0; i < kVals; ++i) v[i] = warp_max(v[i]);
  if (kAllLanes || lane == 0) {
#pragma unroll
    for (int i = 0; i < kVals; ++i) red[(parity * kVals + i) * kGroupWarps + warp] = v[i];
  }
  group_sync(group);
#pragma unroll
  for (int i = 0; i < kVals; ++i) {
    float mx = 0.0f;
#pragma unroll
    for (int q = 0; q < kGroupWarps; q += 4) {
      const float4 r = *reinterpret_cast<const float4*>(&red[(parity * kVals + i) * kGroupWarps + q]);
      mx = fmaxf(mx, fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w)));
    }
    v[i] = mx;
  }
}

// --------------------------------------------------------------------------
// quantize
//
// Signed map: each group stages its full blocks in shared memory one block
// ahead.  While it works on block b, per-thread 16-byte cp.async copies bring
// block b + stride into the group's other 8 KB buffer, and thread 0 asks L2
// for block b + 2 stride.  Every thread copies and later reads the same
// elements (its own slots), so its own cp.async.wait_group orders the two and
// no barrier is needed; the wait is on the thread's own copies, which always
// complete.  The signed code decision costs more instructions per value than
// the unsigned one, and the copies in flight keep DRAM busy meanwhile.  The
// unsigned map loads each block directly (its arithmetic is short enough that
// staging did not pay).  Partial blocks and unaligned inputs are loaded
// element-wise.

constexpr int kQTabBytes = (kTablesBytes + 127) / 128 * 128;          // tables, then the stage
constexpr int kQSmemBytes = kQTabBytes + kQGroups * 2 * BWD_BLOCK * 4;  // + 2 x 8 KB per group

__device__ __forceinline__ void cp_async16(void* smem, const void* src) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(src) : "memory");
}

// Block absmax, codes and stores of one full, aligned block whose 16 values
// per thread are in v.
template <bool kSigned>
__device__ __forceinline__ void quantize_store_vec(const float (&v)[kPer], const bwd::Tables& tab, float* red,
                                                   int parity, int group, int t, int64_t b,
                                                   uint8_t* __restrict__ codes, float* __restrict__ absmax) {
  float mx[1] = {0.0f};
#pragma unroll
  for (int j = 0; j < kPer; j += 2) mx[0] = max3abs(mx[0], v[j], v[j + 1]);
  group_max<1>(mx, red, parity, group, t);
  const float am = mx[0];
  uint32_t w[kQuads];
  quantize_quads<kSigned, true>(v, am, tab, w);
#pragma unroll
  for (int k = 0; k < kQuads; ++k)
    __stcs(reinterpret_cast<unsigned int*>(codes + b * BWD_BLOCK + kSpan * k) + t, w[k]);
  if (t == 0) absmax[b] = am;
}

template <bool kSigned>
__global__ void __launch_bounds__(kQCta, 2)
quantize_kernel(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ codes,
                float* __restrict__ absmax, int vec_ok) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  bwd::Tables& tab = *reinterpret_cast<bwd::Tables*>(smem_raw);
  __shared__ __align__(16) float s_red[kQGroups][2 * kGroupWarps];
  copy_to_smem(&tab, &g_tables, kTablesBytes);
  __syncthreads();

  const int group = threadIdx.x / kGroup, t = threadIdx.x % kGroup;
  const int64_t nb = (n + BWD_BLOCK - 1) / BWD_BLOCK;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kQGroups;
  int it = 0;
  int64_t b = static_cast<int64_t>(blockIdx.x) * kQGroups + group;
  if (kSigned && vec_ok) {  // full blocks through the stage
    const int64_t nfull = n / BWD_BLOCK;
    float* stage = reinterpret_cast<float*>(smem_raw + kQTabBytes) + group * 2 * BWD_BLOCK;
    if (b < nfull) {
#pragma unroll
      for (int k = 0; k < kQuads; ++k) cp_async16(stage + kSpan * k + 4 * t, x + b * BWD_BLOCK + kSpan * k + 4 * t);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (; b < nfull; b += stride, ++it) {
      const int64_t bn = b + stride;
      if (t == 0 && bn + stride < nfull) prefetch_l2(x + (bn + stride) * BWD_BLOCK, 8192u);
      if (bn < nfull) {
        float* nxt = stage + ((it + 1) & 1) * BWD_BLOCK;
#pragma unroll
        for (int k = 0; k < kQuads; ++k) cp_async16(nxt + kSpan * k + 4 * t, x + bn * BWD_BLOCK + kSpan * k + 4 * t);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // this block's copies (the older group)
      const float* cur = stage + (it & 1) * BWD_BLOCK;
      float v[kPer];
#pragma unroll
      for (int k = 0; k < kQuads; ++k) {
        const float4 a = *reinterpret_cast<const float4*>(cur + kSpan * k + 4 * t);
        v[4 * k] = a.x; v[4 * k + 1] = a.y; v[4 * k + 2] = a.z; v[4 * k + 3] = a.w;
      }
      quantize_store_vec<kSigned>(v, tab, s_red[group], it & 1, group, t, b, codes, absmax);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  // direct loads (unsigned map; for the signed map only unaligned inputs and
  // a partial last block remain)
  for (; b < nb; b += stride, ++it) {
    const int64_t base = b * BWD_BLOCK;
    const int rem = static_cast<int>(rem_in_block(n, base));
    const bool vec = vec_ok && rem == BWD_BLOCK;
    if (t == 0 && vec_ok) {  // ask L2 for the group's next block
      const int64_t bn = b + stride;
      if (bn < nb && n - bn * BWD_BLOCK >= BWD_BLOCK) prefetch_l2(x + bn * BWD_BLOCK, 8192u);
    }
    float v[kPer];
    if (vec) {
#pragma unroll
      for (int k = 0; k < kQuads; ++k) {
        const float4 a = ld_stream_f4(x + base + kSpan * k + 4 * t);
        v[4 * k] = a.x; v[4 * k + 1] = a.y; v[4 * k + 2] = a.z; v[4 * k + 3] = a.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int e = slot(t, j);
        v[j] = e < rem ? x[base + e] : 0.0f;  // padding leaves max |x| unchanged
      }
    }
    float mx[1] = {0.0f};
#pragma unroll
    for (int j = 0; j < kPer; j += 2) mx[0] = max3abs(mx[0], v[j], v[j + 1]);
    group_max<1>(mx, s_red[group], it & 1, group, t);
    const float am = mx[0];

    uint32_t w[kQuads];
    quantize_quads<kSigned, true>(v, am, tab, w);
    if (vec) {
#pragma unroll
      for (int k = 0; k < kQuads; ++k) __stcs(reinterpret_cast<unsigned int*>(codes + base + kSpan * k) + t, w[k]);
    } else {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int e = slot(t, j);
        if (e < rem) codes[base + e] = static_cast<uint8_t>(byte_of(w[j >> 2], j & 3));
      }
    }
    if (t == 0) absmax[b] = am;
  }
}

// --------------------------------------------------------------------------
// dequantize (256 threads, 8 elements per thread: 4 t + j and 1024 + 4 t + j)
//
// A full block's 8 KB of output is assembled in shared memory and written by
// one bulk copy (cp.async.bulk, shared -> global) that thread 0 issues; three
// buffers rotate, so up to two blocks' stores are in flight while the next
// block is computed.  Before a buffer is refilled, thread 0 waits until at
// most two bulk groups still read shared memory (cp.async.bulk.wait_group.read:
// a wait on the CTA's own copies, which always complete) and the CTA meets at
// a barrier.  The stream is write-heavy (4 bytes written per byte read); the
// bulk stores reach a higher DRAM rate than per-thread 16-byte stores.
// Partial blocks and unaligned buffers take element-wise stores.

constexpr int kDeqBufs = 3;

template <bool kSigned>
__global__ void __launch_bounds__(kDeqThreads)
dequantize_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ absmax, int64_t n,
                  float* __restrict__ y, int vec_ok) {
  __shared__ __align__(16) float s_map[kCodes];
  __shared__ __align__(128) float s_out[kDeqBufs][BWD_BLOCK];
  copy_to_smem(s_map, g_tables.map[kSigned ? 0 : 1], sizeof(s_map));
  __syncthreads();
  const int tid = threadIdx.x;
  const int64_t nb = (n + BWD_BLOCK - 1) / BWD_BLOCK;
  int buf_i = 0;
  for (int64_t b = blockIdx.x; b < nb; b += gridDim.x) {
    const int64_t base = b * BWD_BLOCK;
    const int rem = static_cast<int>(rem_in_block(n, base));
    const float am = absmax[b];
    if (vec_ok && rem == BWD_BLOCK) {
      float* buf = s_out[buf_i];
      buf_i = (buf_i == kDeqBufs - 1) ? 0 : buf_i + 1;
      if (tid == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kDeqBufs - 1) : "memory");
      __syncthreads();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w = __ldcs(reinterpret_cast<const unsigned int*>(codes + base + 1024 * h) + tid);
        float4 o;
        o.x = __fmul_rn(s_map[byte_of(w, 0)], am);
        o.y = __fmul_rn(s_map[byte_of(w, 1)], am);
        o.z = __fmul_rn(s_map[byte_of(w, 2)], am);
        o.w = __fmul_rn(s_map[byte_of(w, 3)], am);
        reinterpret_cast<float4*>(buf + 1024 * h)[tid] = o;
      }
      // The generic-proxy writes above become visible to the bulk copy.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      if (tid == 0) {
        const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(buf));
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(y + base), "r"(sa),
                     "n"(BWD_BLOCK * 4)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = (j < 4) ? 4 * tid + j : 1024 + 4 * tid + (j - 4);
        if (e < rem) y[base + e] = __fmul_rn(s_map[codes[base + e]], am);
      }
    }
  }
  // Shared memory must outlive the bulk copies that read it.
  if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// --------------------------------------------------------------------------
// state init

__global__ void fill_kernel(uint8_t* __restrict__ a, uint8_t va, uint8_t* __restrict__ b, uint8_t vb,
                            int64_t n, float* __restrict__ fa, float* __restrict__ fb, int64_t nf) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    a[i] = va;
    b[i] = vb;
  }
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nf; i += stride) {
    fa[i] = 0.0f;
    fb[i] = 0.0f;
  }
}



// --------------------------------------------------------------------------
// 8-bit Adam

struct TensorArgs {
  void* p;  // fp32 or bf16 parameters (kernel template argument)
  const void* g;
  uint8_t* mc;
  float* ma;
  uint8_t* vc;
  float* va;
  int64_t n;
  int64_t vec;  // all four element pointers 16-byte aligned
};

struct AdamArgs {
  int64_t block_start[kMaxTensors + 1];  // prefix sums of per-tensor block counts
  TensorArgs t[kMaxTensors];
  int32_t num_tensors;
  float b1, omb1, b2, omb2, eps, step_size, inv_bc2s;
  float decay;  // 1 - lr * weight_decay (decoupled weight decay), 1 for Adam
};

static_assert(sizeof(AdamArgs) <= 32764, "kernel parameter space");

// Element types of parameters and gradients (the values of bwd_dtype).
constexpr int kF32 = BWD_F32, kBF16 = BWD_BF16, kF16 = BWD_F16;

template <int kT>
__host__ __device__ constexpr uint32_t elem_bytes() { return kT == kF32 ? 4u : 2u; }

// Four consecutive elements of type kT widened to fp32 (bf16 and fp16 widen
// exactly).
template <int kT>
__device__ __forceinline__ void load4(const void* base, int64_t e, float* out) {
  if (kT == kF32) {
    const float4 a = ld_stream_f4(static_cast<const float*>(base) + e);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  } else {
    const uint2 a = ld_stream_u2(static_cast<const uint16_t*>(base) + e);
    if (kT == kBF16) {
      out[0] = __uint_as_float(a.x << 16);
      out[1] = __uint_as_float(a.x & 0xffff0000u);
      out[2] = __uint_as_float(a.y << 16);
      out[3] = __uint_as_float(a.y & 0xffff0000u);
    } else {
      out[0] = __half2float(__ushort_as_half(static_cast<unsigned short>(a.x & 0xffffu)));
      out[1] = __half2float(__ushort_as_half(static_cast<unsigned short>(a.x >> 16)));
      out[2] = __half2float(__ushort_as_half(static_cast<unsigned short>(a.y & 0xffffu)));
      out[3] = __half2float(__ushort_as_half(static_cast<unsigned short>(a.y >> 16)));
    }
  }
}

// Branch-free approximate square root and reciprocal (PTX sqrt.approx /
// rcp.approx, a few ulps; a subnormal v counts as 0, which leaves eps alone
// in the denominator).
__device__ __forceinline__ float sqrt_approx(float x) {
  float r;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// One element of type kT, widened to fp32.
template <int kT>
__device__ __forceinline__ float load1(const void* base, int64_t i) {
  if (kT == kF32) return static_cast<const float*>(base)[i];
  const unsigned short h = static_cast<const unsigned short*>(base)[i];
  if (kT == kBF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  return __half2float(__ushort_as_half(h));
}

// 16-bit pattern of x as a bf16 or fp16 value, round to nearest even
// (CUDA's conversions).
template <int kT>
__device__ __forceinline__ uint32_t bits16(float x) {
  if (kT == kBF16) return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
  return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x)));
}

// Two values as a packed pair of bf16 or fp16 values (lo in the low half),
// each rounded to nearest even: one conversion instruction per pair.
template <int kT>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  uint32_t r;
  if (kT == kBF16) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Groups per CTA of the fused step (ms per 7B step).  fp32 parameters with
// bf16 gradients: seven, 13.83 (six 14.55, eight spill more: 14.1-14.6);
// fp32 parameters with fp32 gradients: six, 16.92 (seven 17.33); 16-bit
// parameters: six, bf16 11.69 (seven 12.23, five 12.85 before the split
// block body), fp16 11.73 (seven 12.17).
template <int kG, int kP>
__host__ __device__ constexpr int adam_groups() { return kP == kF32 && kG != kF32 ? 7 : 6; }

// With 16-bit parameters (a step bound by instruction issue) the
// dequantizing lookups read lane-private copies of both maps: entry c of
// map k for lane l sits at byte 256 c + 128 k + 4 l, in bank l, so the 32
// lookups of a warp never share a bank (random codes in one 256-word map
// take about three shared-memory wavefronts per warp lookup: 12.25 against
// 12.67 ms per 7B step), and one byte permute forms the offset
// (code << 8) | (lane << 2) from the code word and the lane's offset (with
// the two maps in separate 32 KB halves, a multiply-add per lookup more:
// 11.35 against 11.46 ms).  The DRAM-bound fp32-parameter step reads the
// maps themselves (with the copies 14.1 against 13.98 ms).  64 KB beside
// the 28 KB of tables; one CTA per SM either way.
constexpr int kLanes = 32;
constexpr int kRepBytes = 2 * bwd::kCodes * kLanes * 4;
template <int kP>
__host__ __device__ constexpr bool adam_rep() { return kP != kF32; }
template <int kP>
__host__ __device__ constexpr int adam_smem() { return kTablesBytes + (adam_rep<kP>() ? kRepBytes : 0); }

// The same two numbers for runtime types (bwd_dtype).
int adam_groups_of(int p_type, int g_type) {
  return p_type == BWD_F32 && g_type != BWD_F32 ? adam_groups<kBF16, kF32>() : adam_groups<kF32, kF32>();
}
int adam_smem_of(int p_type) {
  return p_type == BWD_F32 ? adam_smem<kF32>() : p_type == BWD_BF16 ? adam_smem<kBF16>() : adam_smem<kF16>();
}

// kG: gradient type; kP: parameter type (kF32, kBF16 or kF16; 16-bit
// parameters are widened for the update and rounded back on store).
template <int kG, int kP>
__global__ void __launch_bounds__(kGroup * adam_groups<kG, kP>(), 1)
adam8bit_kernel(const __grid_constant__ AdamArgs args) {
  constexpr int kGroups = adam_groups<kG, kP>();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  bwd::Tables& tab = *reinterpret_cast<bwd::Tables*>(smem_raw);
  float4* rep4 = reinterpret_cast<float4*>(smem_raw + kTablesBytes);
  __shared__ __align__(16) float s_red[kGroups][2 * 2 * kGroupWarps];
  constexpr bool kRep = adam_rep<kP>();
  copy_to_smem(&tab, &g_tables, kTablesBytes);
  __syncthreads();
  if (kRep) {
    for (int i = threadIdx.x; i < kRepBytes / 16; i += blockDim.x) {
      const float v = tab.map[(i >> 3) & 1][i >> 4];  // 256 B per code: 32 lanes of map 0, then of map 1
      rep4[i] = make_float4(v, v, v, v);
    }
    __syncthreads();
  }

  const int group = threadIdx.x / kGroup, t = threadIdx.x % kGroup;
  const int nt = args.num_tensors;
  const int64_t total = args.block_start[nt];
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kGroups;
  int64_t gb = static_cast<int64_t>(blockIdx.x) * kGroups + group;
  if (gb >= total) return;

  // tensor holding global block gb: the last ti with block_start[ti] <= gb
  int lo = 0, hi = nt - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (args.block_start[mid] <= gb) lo = mid; else hi = mid - 1;
  }
  int ti = lo;
  int tn = lo;  // tensor of the block prefetched one iteration ahead (the prefetching threads)

  const float b1 = args.b1, omb1 = args.omb1, b2 = args.b2, omb2 = args.omb2;
  const float eps = args.eps, step_size = args.step_size, inv_bc2s = args.inv_bc2s, decay = args.decay;
  const float* map_s = tab.map[0];
  const float* map_u = tab.map[1];
  const unsigned char* const rep_b = reinterpret_cast<const unsigned char*>(rep4);
  const uint32_t lane4 = (threadIdx.x & (kLanes - 1)) * 4u;

  int it = 0;
  for (; gb < total; gb += stride, ++it) {
    while (args.block_start[ti + 1] <= gb) ++ti;
    const TensorArgs& T = args.t[ti];
    const int64_t lb = gb - args.block_start[ti];
    const int64_t base = lb * BWD_BLOCK;
    const int rem = static_cast<int>(rem_in_block(T.n, base));
    const bool vec = T.vec && rem == BWD_BLOCK;
    const float ma_old = T.ma[lb];
    const float va_old = T.va[lb];
    // the group asks L2 for its next block, so that block's loads find it
    // there instead of in DRAM.  With 16-bit parameters (a step bound by
    // instruction issue) one thread issues the four hints and only a next
    // block in the same tensor is prefetched, which needs no tensor search
    // (13.05 against 13.20 ms per 7B step; one thread instead of four, one
    // array each: 11.47 against 11.69); with fp32 parameters (bound by
    // DRAM) the first block of the next tensor is prefetched too (14.24
    // against 14.31 ms), by one thread with 16-bit gradients (13.58 against
    // 13.82 ms with four) and by four, one array each, with fp32 ones
    // (15.6 against 16.7 ms with one).
    if (kP != kF32) {
      if (t == 0) {
        const int64_t bn = base + stride * BWD_BLOCK;
        if (T.vec && T.n - bn >= BWD_BLOCK) {
          prefetch_l2(static_cast<const char*>(T.p) + bn * elem_bytes<kP>(), BWD_BLOCK * elem_bytes<kP>());
          prefetch_l2(static_cast<const char*>(T.g) + bn * elem_bytes<kG>(), BWD_BLOCK * elem_bytes<kG>());
          prefetch_l2(T.mc + bn, 2048u);
          prefetch_l2(T.vc + bn, 2048u);
        }
      }
    } else if (t < (kG == kF32 ? 4 : 1)) {
      const int64_t gn = gb + stride;
      if (gn < total) {
        while (args.block_start[tn + 1] <= gn) ++tn;
        const TensorArgs& N = args.t[tn];
        const int64_t bn = (gn - args.block_start[tn]) * BWD_BLOCK;
        if (N.vec && N.n - bn >= BWD_BLOCK) {
          if constexpr (kG == kF32) {
            if (t == 0) prefetch_l2(static_cast<const char*>(N.p) + bn * elem_bytes<kP>(), BWD_BLOCK * elem_bytes<kP>());
            else if (t == 1) prefetch_l2(static_cast<const char*>(N.g) + bn * elem_bytes<kG>(), BWD_BLOCK * elem_bytes<kG>());
            else if (t == 2) prefetch_l2(N.mc + bn, 2048u);
            else prefetch_l2(N.vc + bn, 2048u);
          } else {
            prefetch_l2(static_cast<const char*>(N.p) + bn * elem_bytes<kP>(), BWD_BLOCK * elem_bytes<kP>());
            prefetch_l2(static_cast<const char*>(N.g) + bn * elem_bytes<kG>(), BWD_BLOCK * elem_bytes<kG>());
            prefetch_l2(N.mc + bn, 2048u);
            prefetch_l2(N.vc + bn, 2048u);
          }
        }
      }
    }

    // The block's work, compiled twice: for a full block of a tensor whose
    // four arrays are 16-byte aligned (vector loads and stores, no branch on
    // that inside) and for the rest (element-wise, padded).  One branch per
    // block picks the copy; with the three in-body branches of one shared
    // copy the step ran 12.22 against 11.66 ms per 7B step with bf16
    // parameters and 13.96 against 13.83 with fp32 ones.
    auto body = [&](auto vtag) {
      constexpr bool kVec = decltype(vtag)::value;
      float p[kPer], g[kPer];
      uint32_t mw[kQuads], vw[kQuads];
      if constexpr (kVec) {
#pragma unroll
        for (int k = 0; k < kQuads; ++k) {
          const int64_t e = base + kSpan * k + 4 * t;
          load4<kP>(T.p, e, &p[4 * k]);
          load4<kG>(T.g, e, &g[4 * k]);
          mw[k] = ld_stream_u1(T.mc + e);
          vw[k] = ld_stream_u1(T.vc + e);
        }
      } else {
        // padding slots: p = g = 0 and the codes of zero, so m = v = 0 there
        // and the block absmax is unchanged
#pragma unroll
        for (int k = 0; k < kQuads; ++k) {
          uint32_t cm[4], cv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = slot(t, 4 * k + j);
            const bool in = e < rem;
            p[4 * k + j] = in ? load1<kP>(T.p, base + e) : 0.0f;
            g[4 * k + j] = in ? load1<kG>(T.g, base + e) : 0.0f;
            cm[j] = in ? T.mc[base + e] : 128u;
            cv[j] = in ? T.vc[base + e] : 0u;
          }
          mw[k] = pack4(cm[0], cm[1], cm[2], cm[3]);
          vw[k] = pack4(cv[0], cv[1], cv[2], cv[3]);
        }
      }

      // dequantize -> Adam in fp32, two elements at a time.  The moments take
      // one rounding per operation in the oracle's order, so they (and the
      // codes and absmax derived from them) are bit-identical; the parameter
      // update uses branch-free approximate sqrt and reciprocal (a few ulps
      // of the update term)
      float m[kPer], v[kPer];
      float mx[2] = {0.0f, 0.0f};
      const float2 ma2 = bwd::dup2(ma_old), va2 = bwd::dup2(va_old), ic2 = bwd::dup2(inv_bc2s);
      const float2 b1_2 = bwd::dup2(b1), omb1_2 = bwd::dup2(omb1), b2_2 = bwd::dup2(b2), omb2_2 = bwd::dup2(omb2);
      const float2 eps2 = bwd::dup2(eps), nstep2 = bwd::dup2(-step_size), decay2 = bwd::dup2(decay);
#pragma unroll
      for (int j = 0; j < kPer; j += 2) {
        float2 mo, vo;
        if constexpr (kRep) {
          // byte offset (code << 8) | (lane << 2) by one permute
          const uint32_t om0 = __byte_perm(mw[j >> 2], lane4, 0x5504u | ((j & 3) << 4));
          const uint32_t om1 = __byte_perm(mw[j >> 2], lane4, 0x5504u | (((j & 3) + 1) << 4));
          const uint32_t ov0 = __byte_perm(vw[j >> 2], lane4, 0x5504u | ((j & 3) << 4));
          const uint32_t ov1 = __byte_perm(vw[j >> 2], lane4, 0x5504u | (((j & 3) + 1) << 4));
          mo = bwd::mul2(make_float2(*reinterpret_cast<const float*>(rep_b + om0),
                                     *reinterpret_cast<const float*>(rep_b + om1)), ma2);
          vo = bwd::mul2(make_float2(*reinterpret_cast<const float*>(rep_b + 128 + ov0),
                                     *reinterpret_cast<const float*>(rep_b + 128 + ov1)), va2);
        } else {
          const uint32_t im0 = byte_prmt(mw[j >> 2], j & 3), im1 = byte_prmt(mw[j >> 2], (j & 3) + 1);
          const uint32_t iv0 = byte_prmt(vw[j >> 2], j & 3), iv1 = byte_prmt(vw[j >> 2], (j & 3) + 1);
          mo = bwd::mul2(make_float2(map_s[im0], map_s[im1]), ma2);
          vo = bwd::mul2(make_float2(map_u[iv0], map_u[iv1]), va2);
        }
        const float2 g2 = make_float2(g[j], g[j + 1]);
        // products packed, sums scalar: a packed multiply feeding a packed add
        // may be contracted into one fused operation, which would change the
        // rounding
        const float2 bm = bwd::mul2(b1_2, mo), gm = bwd::mul2(omb1_2, g2);
        const float2 bv = bwd::mul2(b2_2, vo), gv = bwd::mul2(bwd::mul2(omb2_2, g2), g2);
        const float2 mm = make_float2(__fadd_rn(bm.x, gm.x), __fadd_rn(bm.y, gm.y));
        const float2 vv = make_float2(__fadd_rn(bv.x, gv.x), __fadd_rn(bv.y, gv.y));
        m[j] = mm.x; m[j + 1] = mm.y; v[j] = vv.x; v[j + 1] = vv.y;
        const float2 den = bwd::fma2(make_float2(sqrt_approx(vv.x), sqrt_approx(vv.y)), ic2, eps2);
        const float2 rc = make_float2(rcp_approx(den.x), rcp_approx(den.y));
        const float2 pp = bwd::fma2(bwd::mul2(nstep2, mm), rc, bwd::mul2(make_float2(p[j], p[j + 1]), decay2));
        p[j] = pp.x; p[j + 1] = pp.y;
        mx[0] = max3abs(mx[0], mm.x, mm.y);
        mx[1] = max3(mx[1], vv.x, vv.y);
      }
      if constexpr (kVec) {
#pragma unroll
        for (int k = 0; k < kQuads; ++k) {
          const int64_t e = base + kSpan * k + 4 * t;
          if (kP != kF32)
            __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(T.p) + e),
                   make_uint2(pack16<kP>(p[4 * k], p[4 * k + 1]), pack16<kP>(p[4 * k + 2], p[4 * k + 3])));
          else
            __stcs(reinterpret_cast<float4*>(static_cast<float*>(T.p) + e),
                   make_float4(p[4 * k], p[4 * k + 1], p[4 * k + 2], p[4 * k + 3]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int e = slot(t, j);
          if (e < rem) {
            if (kP != kF32) static_cast<uint16_t*>(T.p)[base + e] = static_cast<uint16_t>(bits16<kP>(p[j]));
            else static_cast<float*>(T.p)[base + e] = p[j];
          }
        }
      }

      // block absmax of the new moments, then requantize
      group_max<2, kP != kF32>(mx, s_red[group], it & 1, group, t);
      const float am = mx[0], av = mx[1];
      quantize_quads<true, false>(m, am, tab, mw);
      quantize_quads<false, false>(v, av, tab, vw);
      if constexpr (kVec) {
#pragma unroll
        for (int k = 0; k < kQuads; ++k) {
          __stcs(reinterpret_cast<unsigned int*>(T.mc + base + kSpan * k) + t, mw[k]);
          __stcs(reinterpret_cast<unsigned int*>(T.vc + base + kSpan * k) + t, vw[k]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int e = slot(t, j);
          if (e < rem) {
            T.mc[base + e] = static_cast<uint8_t>(byte_of(mw[j >> 2], j & 3));
            T.vc[base + e] = static_cast<uint8_t>(byte_of(vw[j >> 2], j & 3));
          }
        }
      }
      // every thread of the group read the old absmax before the barrier above
      if (t == 0) { T.ma[lb] = am; T.va[lb] = av; }
    };
    if (vec) body(std::true_type{});
    else body(std::false_type{});
  }
}

// --------------------------------------------------------------------------
// host side

}  // namespace

namespace bwd {
namespace host {

namespace {
thread_local std::string t_last_error;
}  // namespace

bwd_status fail(bwd_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

bwd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(BWD_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bwd_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, what);
  return BWD_OK;
}

const char* last_error() { return t_last_error.c_str(); }

namespace {
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);  // CUresult cuCtxGetId(CUcontext, ...)
std::once_flag g_ctx_fn_once;
CtxGetIdFn g_ctx_fn = nullptr;
}  // namespace

bwd_status current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_fn_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_fn = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!g_ctx_fn) return fail(BWD_ERR_CUDA, "the driver does not provide cuCtxGetId");
  if (g_ctx_fn(nullptr, id) == 0) return BWD_OK;
  // no current context yet: make the current device's primary context current
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  if (g_ctx_fn(nullptr, id) != 0) return fail(BWD_ERR_CUDA, "cuCtxGetId failed for the current context");
  return BWD_OK;
}

}  // namespace host
}  // namespace bwd

namespace {

using bwd::host::aligned16;
using bwd::host::aligned_to;
using bwd::host::check_launch;
using bwd::host::cuda_fail;
using bwd::host::fail;

struct DeviceState {
  bool ready = false;
  unsigned long long ctx = 0;  // context the tables were uploaded to
  int num_sms = 0;
  int occ_quant[2] = {0, 0};
  int occ_dequant[2] = {0, 0};
  int occ_adam[9] = {};  // [3 * parameter type + gradient type]
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
bwd::Tables g_host_tables;
bool g_host_built = false;

// Opts a kernel into `smem` bytes of dynamic shared memory and returns how
// many of its CTAs fit on one SM.
bwd_status occupancy(const void* fn, int threads, int smem, int* out) {
  int v = 0;
  cudaError_t e;
  if (smem > 0) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)");
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, threads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  *out = v > 0 ? v : 1;
  return BWD_OK;
}

// Uploads the tables to the current device once and caches launch limits.
bwd_status ensure_device(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(BWD_ERR_CUDA, "device ordinal %d unsupported", dev);
  unsigned long long ctx = 0;
  bwd_status s = bwd::host::current_context_id(&ctx);
  if (s != BWD_OK) return s;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.ready && d.ctx == ctx) { *out = &d; return BWD_OK; }
  d.ready = false;  // first use, or a new context (its __device__ tables start zeroed)
  if (!g_host_built) {
    char err[128] = {0};
    if (bwd::build_tables(&g_host_tables, err, sizeof err) != 0)
      return fail(BWD_ERR_CUDA, "code table build failed: %s", err);
    g_host_built = true;
  }
  e = cudaMemcpyToSymbol(g_tables, &g_host_tables, sizeof(bwd::Tables));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(tables)");
  e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  const void* kq[2] = {reinterpret_cast<const void*>(quantize_kernel<true>),
                       reinterpret_cast<const void*>(quantize_kernel<false>)};
  const void* kd[2] = {reinterpret_cast<const void*>(dequantize_kernel<true>),
                       reinterpret_cast<const void*>(dequantize_kernel<false>)};
  const void* ka[9] = {
      reinterpret_cast<const void*>(adam8bit_kernel<kF32, kF32>), reinterpret_cast<const void*>(adam8bit_kernel<kBF16, kF32>),
      reinterpret_cast<const void*>(adam8bit_kernel<kF16, kF32>), reinterpret_cast<const void*>(adam8bit_kernel<kF32, kBF16>),
      reinterpret_cast<const void*>(adam8bit_kernel<kBF16, kBF16>), reinterpret_cast<const void*>(adam8bit_kernel<kF16, kBF16>),
      reinterpret_cast<const void*>(adam8bit_kernel<kF32, kF16>), reinterpret_cast<const void*>(adam8bit_kernel<kBF16, kF16>),
      reinterpret_cast<const void*>(adam8bit_kernel<kF16, kF16>)};
  for (int k = 0; k < 2; ++k) {
    if ((s = occupancy(kq[k], kQCta, k == 0 ? kQSmemBytes : kTablesBytes, &d.occ_quant[k])) != BWD_OK) return s;
    if ((s = occupancy(kd[k], kDeqThreads, 0, &d.occ_dequant[k])) != BWD_OK) return s;
  }
  for (int k = 0; k < 9; ++k)
    if ((s = occupancy(ka[k], kGroup * adam_groups_of(k / 3, k % 3), adam_smem_of(k / 3), &d.occ_adam[k])) != BWD_OK)
      return s;
  d.ctx = ctx;
  d.ready = true;
  *out = &d;
  return BWD_OK;
}


// CTAs for `blocks` quantization blocks when each CTA works on `per_cta` at a
// time: enough to cover them, at most one full wave of resident CTAs.
int grid_for(int64_t blocks, int per_cta, const DeviceState& d, int occ) {
  const int64_t need = (blocks + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(d.num_sms) * occ;
  return static_cast<int>(need < cap ? need : cap);
}


bool valid_kind(bwd_map_kind k) { return k == BWD_MAP_SIGNED || k == BWD_MAP_UNSIGNED; }

bwd_status check_hparams(const bwd_adam_hparams* hp) {
  if (!hp) return fail(BWD_ERR_INVALID_ARG, "hparams is NULL");
  if (hp->step < 1) return fail(BWD_ERR_INVALID_ARG, "step must be >= 1 (got %lld)", (long long)hp->step);
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->eps) || hp->eps < 0.0f)
    return fail(BWD_ERR_INVALID_ARG, "lr and eps must be finite, eps >= 0");
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return fail(BWD_ERR_INVALID_ARG, "betas must lie in [0, 1)");
  if (!std::isfinite(hp->weight_decay) || hp->weight_decay < 0.0f)
    return fail(BWD_ERR_INVALID_ARG, "weight_decay must be finite and >= 0");
  return BWD_OK;
}

// Host scalars of the update: bias corrections in binary64, rounded once.
void fill_scalars(const bwd_adam_hparams* hp, AdamArgs* a) {
  const double b1 = hp->beta1, b2 = hp->beta2, t = static_cast<double>(hp->step);
  const double bc1 = 1.0 - std::pow(b1, t);
  const double bc2 = 1.0 - std::pow(b2, t);
  a->b1 = hp->beta1;
  a->b2 = hp->beta2;
  a->omb1 = static_cast<float>(1.0 - b1);
  a->omb2 = static_cast<float>(1.0 - b2);
  a->eps = hp->eps;
  a->step_size = static_cast<float>(static_cast<double>(hp->lr) / bc1);
  a->inv_bc2s = static_cast<float>(1.0 / std::sqrt(bc2));
  a->decay = static_cast<float>(1.0 - static_cast<double>(hp->lr) * static_cast<double>(hp->weight_decay));
}

template <int kG, int kP>
void launch_typed(const AdamArgs& a, int grid, cudaStream_t st) {
  adam8bit_kernel<kG, kP><<<grid, kGroup * adam_groups<kG, kP>(), adam_smem<kP>(), st>>>(a);
}

bwd_status launch_adam_chunk(const AdamArgs& a, int g_type, int p_type, const DeviceState& d, cudaStream_t st) {
  const int64_t total = a.block_start[a.num_tensors];
  if (total == 0) return BWD_OK;
  const int grid = grid_for(total, adam_groups_of(p_type, g_type), d, d.occ_adam[3 * p_type + g_type]);
  switch (3 * p_type + g_type) {
    case 0: launch_typed<kF32, kF32>(a, grid, st); break;
    case 1: launch_typed<kBF16, kF32>(a, grid, st); break;
    case 2: launch_typed<kF16, kF32>(a, grid, st); break;
    case 3: launch_typed<kF32, kBF16>(a, grid, st); break;
    case 4: launch_typed<kBF16, kBF16>(a, grid, st); break;
    case 5: launch_typed<kF16, kBF16>(a, grid, st); break;
    case 6: launch_typed<kF32, kF16>(a, grid, st); break;
    case 7: launch_typed<kBF16, kF16>(a, grid, st); break;
    default: launch_typed<kF16, kF16>(a, grid, st); break;
  }
  return check_launch("adam8bit_kernel launch");
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI

extern "C" {

const char* bwd_status_string(bwd_status s) {
  switch (s) {
    case BWD_OK: return "ok";
    case BWD_ERR_INVALID_ARG: return "invalid argument";
    case BWD_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case BWD_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* bwd_last_error(void) { return bwd::host::last_error(); }

bwd_status bwd_init(void) {
  DeviceState* d = nullptr;
  return ensure_device(&d);
}

bwd_status bwd_quantize_blockwise(const float* x, int64_t n, bwd_map_kind kind, uint8_t* codes,
                                  float* absmax, void* stream) {
  if (n < 0) return fail(BWD_ERR_INVALID_ARG, "n < 0");
  if (!valid_kind(kind)) return fail(BWD_ERR_INVALID_ARG, "bad map kind %d", (int)kind);
  if (n == 0) return BWD_OK;
  if (!x || !codes || !absmax) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned_to(x, 4) || !aligned_to(absmax, 4)) return fail(BWD_ERR_INVALID_ARG, "fp32 pointer not 4-byte aligned");
  DeviceState* d = nullptr;
  bwd_status s = ensure_device(&d);
  if (s != BWD_OK) return s;
  const int64_t nb = bwd_num_blocks(n);
  const int vec = aligned16(x) && aligned16(codes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kind == BWD_MAP_SIGNED)
    quantize_kernel<true><<<grid_for(nb, kQGroups, *d, d->occ_quant[0]), kQCta, kQSmemBytes, st>>>(
        x, n, codes, absmax, vec);
  else
    quantize_kernel<false><<<grid_for(nb, kQGroups, *d, d->occ_quant[1]), kQCta, kTablesBytes, st>>>(
        x, n, codes, absmax, vec);
  return check_launch("quantize_kernel launch");
}

bwd_status bwd_dequantize_blockwise(const uint8_t* codes, const float* absmax, int64_t n,
                                    bwd_map_kind kind, float* y, void* stream) {
  if (n < 0) return fail(BWD_ERR_INVALID_ARG, "n < 0");
  if (!valid_kind(kind)) return fail(BWD_ERR_INVALID_ARG, "bad map kind %d", (int)kind);
  if (n == 0) return BWD_OK;
  if (!codes || !absmax || !y) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned_to(absmax, 4) || !aligned_to(y, 4)) return fail(BWD_ERR_INVALID_ARG, "fp32 pointer not 4-byte aligned");
  DeviceState* d = nullptr;
  bwd_status s = ensure_device(&d);
  if (s != BWD_OK) return s;
  const int64_t nb = bwd_num_blocks(n);
  const int vec = aligned16(codes) && aligned16(y);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kind == BWD_MAP_SIGNED)
    dequantize_kernel<true><<<grid_for(nb, 1, *d, d->occ_dequant[0]), kDeqThreads, 0, st>>>(
        codes, absmax, n, y, vec);
  else
    dequantize_kernel<false><<<grid_for(nb, 1, *d, d->occ_dequant[1]), kDeqThreads, 0, st>>>(
        codes, absmax, n, y, vec);
  return check_launch("dequantize_kernel launch");
}

bwd_status bwd_state_init(uint8_t* m_codes, float* m_absmax, uint8_t* v_codes, float* v_absmax,
                          int64_t n, void* stream) {
  if (n < 0) return fail(BWD_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return BWD_OK;
  if (!m_codes || !m_absmax || !v_codes || !v_absmax) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned_to(m_absmax, 4) || !aligned_to(v_absmax, 4))
    return fail(BWD_ERR_INVALID_ARG, "fp32 pointer not 4-byte aligned");
  DeviceState* d = nullptr;
  bwd_status s = ensure_device(&d);
  if (s != BWD_OK) return s;
  const int64_t work = (n + kDeqThreads - 1) / kDeqThreads;
  const int grid = static_cast<int>(work < d->num_sms * 8 ? work : d->num_sms * 8);
  fill_kernel<<<grid, kDeqThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      m_codes, 128, v_codes, 0, n, m_absmax, v_absmax, bwd_num_blocks(n));
  return check_launch("fill_kernel launch");
}

}  // extern "C"

namespace {

// Shared body of the multi-tensor entry points; PP is float* const* or
// void* const* (the parameter pointers).
template <typename PP>
bwd_status step_multi(int32_t num_tensors, PP p, bwd_dtype p_dtype, const void* const* g, bwd_dtype g_dtype,
                      uint8_t* const* m_codes, float* const* m_absmax, uint8_t* const* v_codes,
                      float* const* v_absmax, const int64_t* n, const bwd_adam_hparams* hp, void* stream) {
  if (num_tensors < 0) return fail(BWD_ERR_INVALID_ARG, "num_tensors < 0");
  if (g_dtype != BWD_F32 && g_dtype != BWD_BF16 && g_dtype != BWD_F16)
    return fail(BWD_ERR_UNSUPPORTED_DTYPE, "gradient dtype %d", (int)g_dtype);
  if (p_dtype != BWD_F32 && p_dtype != BWD_BF16 && p_dtype != BWD_F16)
    return fail(BWD_ERR_UNSUPPORTED_DTYPE, "parameter dtype %d", (int)p_dtype);
  bwd_status s = check_hparams(hp);
  if (s != BWD_OK) return s;
  if (num_tensors == 0) return BWD_OK;
  if (!p || !g || !m_codes || !m_absmax || !v_codes || !v_absmax || !n)
    return fail(BWD_ERR_INVALID_ARG, "NULL array");
  bool any_work = false;
  for (int32_t i = 0; i < num_tensors; ++i) {
    if (n[i] < 0) return fail(BWD_ERR_INVALID_ARG, "tensor %d: n < 0", i);
    if (n[i] > 0 && (!p[i] || !g[i] || !m_codes[i] || !m_absmax[i] || !v_codes[i] || !v_absmax[i]))
      return fail(BWD_ERR_INVALID_ARG, "tensor %d: NULL pointer", i);
    if (n[i] > 0 && (!aligned_to(p[i], p_dtype == BWD_F32 ? 4 : 2) || !aligned_to(g[i], g_dtype == BWD_F32 ? 4 : 2) ||
                     !aligned_to(m_absmax[i], 4) || !aligned_to(v_absmax[i], 4)))
      return fail(BWD_ERR_INVALID_ARG, "tensor %d: pointer not aligned to its element size", i);
    any_work = any_work || n[i] > 0;
  }
  if (!any_work) return BWD_OK;
  DeviceState* d = nullptr;
  if ((s = ensure_device(&d)) != BWD_OK) return s;

  static thread_local AdamArgs a;  // ~32 KB: kept off the stack
  fill_scalars(hp, &a);
  const int g_type = static_cast<int>(g_dtype), p_type = static_cast<int>(p_dtype);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int k = 0;
  a.block_start[0] = 0;
  for (int32_t i = 0; i < num_tensors; ++i) {
    if (n[i] == 0) continue;
    TensorArgs& t = a.t[k];
    t.p = p[i];
    t.g = g[i];
    t.mc = m_codes[i];
    t.ma = m_absmax[i];
    t.vc = v_codes[i];
    t.va = v_absmax[i];
    t.n = n[i];
    t.vec = aligned16(p[i]) && aligned16(g[i]) && aligned16(m_codes[i]) && aligned16(v_codes[i]);
    a.block_start[k + 1] = a.block_start[k] + bwd_num_blocks(n[i]);
    ++k;
    if (k == kMaxTensors) {
      a.num_tensors = k;
      if ((s = launch_adam_chunk(a, g_type, p_type, *d, st)) != BWD_OK) return s;
      k = 0;
      a.block_start[0] = 0;
    }
  }
  if (k > 0) {
    a.num_tensors = k;
    if ((s = launch_adam_chunk(a, g_type, p_type, *d, st)) != BWD_OK) return s;
  }
  return BWD_OK;
}

}  // namespace

extern "C" {

bwd_status bwd_adam8bit_step_multi(int32_t num_tensors, float* const* p, const void* const* g,
                                   bwd_dtype g_dtype, uint8_t* const* m_codes, float* const* m_absmax,
                                   uint8_t* const* v_codes, float* const* v_absmax, const int64_t* n,
                                   const bwd_adam_hparams* hp, void* stream) {
  return step_multi(num_tensors, p, BWD_F32, g, g_dtype, m_codes, m_absmax, v_codes, v_absmax, n, hp, stream);
}

bwd_status bwd_adam8bit_step_multi_ex(int32_t num_tensors, void* const* p, bwd_dtype p_dtype,
                                      const void* const* g, bwd_dtype g_dtype, uint8_t* const* m_codes,
                                      float* const* m_absmax, uint8_t* const* v_codes,
                                      float* const* v_absmax, const int64_t* n,
                                      const bwd_adam_hparams* hp, void* stream) {
  return step_multi(num_tensors, p, p_dtype, g, g_dtype, m_codes, m_absmax, v_codes, v_absmax, n, hp, stream);
}

bwd_status bwd_adam8bit_step(float* p, const void* g, bwd_dtype g_dtype, uint8_t* m_codes,
                             float* m_absmax, uint8_t* v_codes, float* v_absmax, int64_t n,
                             const bwd_adam_hparams* hp, void* stream) {
  return bwd_adam8bit_step_multi(1, &p, &g, g_dtype, &m_codes, &m_absmax, &v_codes, &v_absmax, &n, hp,
                                 stream);
}

}  // extern "C"
