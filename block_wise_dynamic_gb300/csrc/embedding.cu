// sm_103a kernels and C ABI of the stable embedding layer.
//
// Method: "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (summary on
// wiki.neutronadmin.com/news/16836), section 二 / 稳定的词嵌入层: the
// embedding weight starts from a Xavier-uniform draw, and a layer
// normalisation follows the lookup so that the layer's output has variance
// close to 1.  Readings: the Xavier bound is b = sqrt(6 / (V + D)) for a
// (V, D) weight; the normalisation is LayerNorm over D with biased variance
// and a learnable scale gamma and shift beta; the backward pass is the
// gradient of that map, accumulated into the weight rows of the tokens.
//
// Work decomposition.  Forward: a group of 128 threads owns one token (one
// row of D fp32 values) at a time and walks the tokens with a grid stride.
// On the fast path (D a multiple of 4 and at most 4096, every row pointer
// 16-byte aligned) thread t of a group holds the float4 chunks t, t + 128,
// ... of the row in registers, so a row is read from HBM once: every warp
// access is one contiguous 512-byte span.  Row statistics are sums over the
// group (warp shuffles, then the group's warp partials through shared memory
// in a fixed order, so results do not depend on scheduling): mean, then the
// centred sum of squares from the registers, then
// y = (x - mean) rstd gamma + beta.  Thread 0 asks L2 for the group's next
// row meanwhile (cp.async.bulk.prefetch.L2).
//
// Backward, fast path: for one vocabulary row the layer's gradient is linear
// in dL/dy, so the tokens of a row need only the sum S of their dL/dy rows
// (one LayerNorm backward per run of equal ids instead of one per token, and
// one atomic add of the row's dx per run).  One CTA per SM sorts a chunk of
// consecutive tokens by id in shared memory; a producer warp streams the
// run's dL/dy rows and then its weight row into a ring of shared-memory
// slots (cp.async.bulk with full / empty mbarriers), sixteen consumer warps
// sum the run in registers, reduce the two row sums once and add
// dx = rstd (G - mean(G) - xhat mean(G xhat)), G = S gamma, into the weight
// row's gradient with vector atomics; each consumer keeps dgamma and dbeta
// partials for its columns and adds them once at the end.  Other shapes take
// a per-element path with the same arithmetic, token by token.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "bwd.h"
#include "exact_div.cuh"  // packed binary32 pair arithmetic (add2, mul2, fma2)
#include "host_util.h"

namespace {

using bwd::host::aligned16;
using bwd::host::aligned_to;
using bwd::host::check_launch;
using bwd::host::cuda_fail;
using bwd::host::fail;

constexpr int kGroup = 128;                       // threads per token
constexpr int kGroupWarps = kGroup / 32;          // 4
constexpr int kChunks = 8;                        // float4 chunks per thread on the fast path
constexpr int kFastMaxDim = kGroup * 4 * kChunks; // 4096
constexpr int kFwdGroups = 2;                     // forward CTA: 256 threads
constexpr int kSlowGroups = 2;                    // per-element path: 256 threads
constexpr int kInitThreads = 256;
constexpr int kMaxDevices = 64;

// --------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Named barrier of one 128-thread group (barrier 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "n"(kGroup) : "memory");
}

// Sums of kVals values over the 128 threads of a group; every thread gets
// the results.  `red` is the group's [2 slots][kVals][4 warps] scratch; the
// slot alternates between consecutive calls, so a thread that runs ahead
// never overwrites partials another thread has yet to read.
template <int kVals>
__device__ __forceinline__ void group_sum(float (&v)[kVals], float* red, int slot, int group, int t) {
  const int lane = t & 31, warp = t >> 5;
#pragma unroll
  for (int i = 0; i < kVals; ++i) v[i] = warp_sum(v[i]);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kVals; ++i) red[(slot * kVals + i) * kGroupWarps + warp] = v[i];
  }
  group_sync(group);
#pragma unroll
  for (int i = 0; i < kVals; ++i) {
    const float4 r = *reinterpret_cast<const float4*>(&red[(slot * kVals + i) * kGroupWarps]);
    v[i] = __fadd_rn(__fadd_rn(r.x, r.y), __fadd_rn(r.z, r.w));
  }
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Hint: bring `bytes` (a multiple of 16, 16-byte aligned) of global memory
// into L2.  Nothing waits for it, so it cannot stall or hang anything.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void red_add4(float* p, float4 v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// --------------------------------------------------------------------------
// Xavier-uniform initialisation: w = (2 u - 1) b, u = (r >> 8) 2^-24.  The
// integer converts exactly, 2 u - 1 is exact (a multiple of 2^-23 in
// [-1, 1)), so the product with the binary32 bound is the one rounding.

__global__ void __launch_bounds__(kInitThreads)
embed_init_kernel(const uint32_t* __restrict__ words, int64_t n, float bound, float* __restrict__ w) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float u = __fmul_rn(static_cast<float>(words[i] >> 8), 0x1p-24f);
    w[i] = __fmul_rn(__fsub_rn(__fmul_rn(2.0f, u), 1.0f), bound);
  }
}

// --------------------------------------------------------------------------
// forward: y = LayerNorm(weight[id]); mean and rstd per token (optional).
// A token id outside [0, V) gives a row of NaN (row 0 is read instead, so
// no access leaves the weight).

__global__ void __launch_bounds__(kGroup * kFwdGroups, 3)
embed_fwd_kernel(const int64_t* __restrict__ ids, int64_t num_tokens, const float* __restrict__ w, int64_t vocab,
                 int dim, const float* __restrict__ gamma, const float* __restrict__ beta, float eps,
                 float* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd) {
  __shared__ __align__(16) float s_red[kFwdGroups][2 * kGroupWarps];
  const int group = threadIdx.x / kGroup, t = threadIdx.x % kGroup;
  const int nch = dim >> 2;
  const float fdim = static_cast<float>(dim);
  const float qnan = __int_as_float(0x7fc00000);
  int slot = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kFwdGroups;
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * kFwdGroups + group; tok < num_tokens; tok += stride) {
    const int64_t id = ids[tok];
    const bool ok = id >= 0 && id < vocab;
    const float* row = w + (ok ? id : 0) * static_cast<int64_t>(dim);
    if (t == 0 && tok + stride < num_tokens) {  // L2 fetches the group's next row meanwhile
      const int64_t nid = ids[tok + stride];
      prefetch_l2(w + ((nid >= 0 && nid < vocab) ? nid : 0) * static_cast<int64_t>(dim),
                  static_cast<uint32_t>(dim * 4));
    }
    float4 x[kChunks];
    float s[1] = {0.0f};
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
      const int c = t + kGroup * k;
      if (c < nch) {
        x[k] = ld4(row + 4 * c);
        s[0] = __fadd_rn(s[0], __fadd_rn(__fadd_rn(x[k].x, x[k].y), __fadd_rn(x[k].z, x[k].w)));
      } else {
        x[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
    group_sum<1>(s, s_red[group], slot, group, t);
    slot ^= 1;
    const float mu = __fdiv_rn(s[0], fdim);
    float q[1] = {0.0f};
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
      if (t + kGroup * k < nch) {
        x[k].x = __fsub_rn(x[k].x, mu);
        x[k].y = __fsub_rn(x[k].y, mu);
        x[k].z = __fsub_rn(x[k].z, mu);
        x[k].w = __fsub_rn(x[k].w, mu);
        q[0] = __fadd_rn(q[0], __fadd_rn(__fadd_rn(__fmul_rn(x[k].x, x[k].x), __fmul_rn(x[k].y, x[k].y)),
                                         __fadd_rn(__fmul_rn(x[k].z, x[k].z), __fmul_rn(x[k].w, x[k].w))));
      }
    }
    group_sum<1>(q, s_red[group], slot, group, t);
    slot ^= 1;
    const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(q[0], fdim), eps));
    float* yrow = y + tok * static_cast<int64_t>(dim);
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
      const int c = t + kGroup * k;
      if (c < nch) {
        const float4 g = ldg4(gamma + 4 * c), b = ldg4(beta + 4 * c);
        float4 o;
        o.x = __fadd_rn(__fmul_rn(__fmul_rn(x[k].x, r), g.x), b.x);
        o.y = __fadd_rn(__fmul_rn(__fmul_rn(x[k].y, r), g.y), b.y);
        o.z = __fadd_rn(__fmul_rn(__fmul_rn(x[k].z, r), g.z), b.z);
        o.w = __fadd_rn(__fmul_rn(__fmul_rn(x[k].w, r), g.w), b.w);
        if (!ok) o = make_float4(qnan, qnan, qnan, qnan);
        __stcs(reinterpret_cast<float4*>(yrow + 4 * c), o);
      }
    }
    if (t == 0) {
      if (mean) mean[tok] = ok ? mu : qnan;
      if (rstd) rstd[tok] = ok ? r : qnan;
    }
  }
}

// Any D and alignment: one element per thread per step, the row re-read
// from L1/L2 for each pass.
__global__ void __launch_bounds__(kGroup * kSlowGroups)
embed_fwd_slow_kernel(const int64_t* __restrict__ ids, int64_t num_tokens, const float* __restrict__ w,
                      int64_t vocab, int64_t dim, const float* __restrict__ gamma, const float* __restrict__ beta,
                      float eps, float* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd) {
  __shared__ __align__(16) float s_red[kSlowGroups][2 * kGroupWarps];
  const int group = threadIdx.x / kGroup, t = threadIdx.x % kGroup;
  const float fdim = static_cast<float>(dim);
  const float qnan = __int_as_float(0x7fc00000);
  int slot = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kSlowGroups;
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * kSlowGroups + group; tok < num_tokens; tok += stride) {
    const int64_t id = ids[tok];
    const bool ok = id >= 0 && id < vocab;
    const float* row = w + (ok ? id : 0) * dim;
    float s[1] = {0.0f};
    for (int64_t j = t; j < dim; j += kGroup) s[0] = __fadd_rn(s[0], row[j]);
    group_sum<1>(s, s_red[group], slot, group, t);
    slot ^= 1;
    const float mu = __fdiv_rn(s[0], fdim);
    float q[1] = {0.0f};
    for (int64_t j = t; j < dim; j += kGroup) {
      const float d = __fsub_rn(row[j], mu);
      q[0] = __fadd_rn(q[0], __fmul_rn(d, d));
    }
    group_sum<1>(q, s_red[group], slot, group, t);
    slot ^= 1;
    const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(q[0], fdim), eps));
    float* yrow = y + tok * dim;
    for (int64_t j = t; j < dim; j += kGroup)
      yrow[j] = ok ? __fadd_rn(__fmul_rn(__fmul_rn(__fsub_rn(row[j], mu), r), gamma[j]), beta[j]) : qnan;
    if (t == 0) {
      if (mean) mean[tok] = ok ? mu : qnan;
      if (rstd) rstd[tok] = ok ? r : qnan;
    }
  }
}

// --------------------------------------------------------------------------
// backward: dweight[id] += dx, dgamma += dy xhat, dbeta += dy (accumulated).
// Tokens whose id lies outside [0, V) are skipped.

__global__ void __launch_bounds__(kGroup * kSlowGroups)
embed_bwd_slow_kernel(const int64_t* __restrict__ ids, int64_t num_tokens, const float* __restrict__ w,
                      int64_t vocab, int64_t dim, const float* __restrict__ gamma, const float* __restrict__ mean,
                      const float* __restrict__ rstd, const float* __restrict__ dy, float* __restrict__ dw,
                      float* __restrict__ dgamma, float* __restrict__ dbeta) {
  __shared__ __align__(16) float s_red[kSlowGroups][2 * 2 * kGroupWarps];
  const int group = threadIdx.x / kGroup, t = threadIdx.x % kGroup;
  const float fdim = static_cast<float>(dim);
  int slot = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kSlowGroups;
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * kSlowGroups + group; tok < num_tokens; tok += stride) {
    const int64_t id = ids[tok];
    if (id < 0 || id >= vocab) continue;
    const float mu = mean[tok], r = rstd[tok];
    const float* row = w + id * dim;
    const float* drow = dy + tok * dim;
    float s[2] = {0.0f, 0.0f};
    for (int64_t j = t; j < dim; j += kGroup) {
      const float xh = __fmul_rn(__fsub_rn(row[j], mu), r);
      const float gg = __fmul_rn(drow[j], gamma[j]);
      s[0] = __fadd_rn(s[0], gg);
      s[1] = __fadd_rn(s[1], __fmul_rn(gg, xh));
    }
    group_sum<2>(s, s_red[group], slot, group, t);
    slot ^= 1;
    const float m1 = __fdiv_rn(s[0], fdim), m2 = __fdiv_rn(s[1], fdim);
    for (int64_t j = t; j < dim; j += kGroup) {
      const float xh = __fmul_rn(__fsub_rn(row[j], mu), r);
      const float d = drow[j];
      atomicAdd(dw + id * dim + j, __fmul_rn(r, __fsub_rn(__fsub_rn(__fmul_rn(d, gamma[j]), m1), __fmul_rn(xh, m2))));
      atomicAdd(dgamma + j, __fmul_rn(d, xh));
      atomicAdd(dbeta + j, d);
    }
  }
}

// --------------------------------------------------------------------------
// mbarrier and bulk-copy helpers of the backward's fast path and of the
// bounded-wait self-test.  Every wait is bounded: after about a second (or
// 2^24 polls) it gives up and g_embed_fault is set (read and cleared by
// bwd_check_device).
__device__ unsigned int g_embed_fault;  // set when a bounded wait gives up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
               " selp.u32 %0, 1, 0, p;\n}" : "=r"(done) : "r"(a), "r"(parity) : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __noinline__ bool mbar_wait_slow(uint32_t a, uint32_t parity) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 24); ++i) {
    if (mbar_try(a, parity)) return true;
    if (global_ns() - t0 > 1000000000ull) return false;
  }
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  return mbar_try(a, parity) || mbar_wait_slow(a, parity);
}

// Backward by runs of equal ids.  For one vocabulary row the gradient of
// the layer is linear in dL/dy (x, mean and rstd are the row's), so the
// tokens of that row need only the sum S of their dL/dy rows: one LayerNorm
// backward on S gives the row's summed dx, and S xhat and S are its shares of
// dgamma and dbeta.  Each CTA (one per SM) takes a chunk of consecutive
// tokens, sorts its (id, position) pairs in shared memory, and walks the
// runs of equal ids in ascending id order.  Two consumer groups of seven
// warps take alternate runs, so one group's row reduction overlaps the other
// group's streaming; each group has its own ring of shared-memory slots and
// its own producer warp, which copies the group's runs, each run's dL/dy rows
// and then its weight row, into the ring (cp.async.bulk; a "full" mbarrier
// per slot counts the bytes, an "empty" one the consumer warps that released
// it; one consumer per ring, so every wait is on the slot's next phase).  A
// group adds the run's dL/dy rows into S in registers,
// and at the weight row reduces the two row sums once and adds dx into the
// row's gradient with vector atomics (other chunks may hold the same id).
// Every CTA visits ids in ascending order, so a row that several SMs touch
// is touched at about the same time and stays in L2; the streamed dL/dy rows
// are copied with an L2 evict-first policy.
//
// Every wait is bounded (about a second, or 2^24 polls).  A wait that gives
// up sets the device fault word and the CTA's fail flag; from then on every
// wait of the CTA returns at once and the producer issues no more copies, so
// all threads run the same barriers to the end; before the CTA exits, the
// producers wait (bounded) for the last copy they issued into each slot.
constexpr int kRGroups = 2;                          // consumer groups, alternate runs
constexpr int kRGT = 224;                            // threads per consumer group (7 warps)
constexpr int kRGWarps = kRGT / 32;
constexpr int kRCons = kRGroups * kRGT;
constexpr int kRThreads = kRCons + 32 * kRGroups;    // + a producer warp per group: 16 warps, 128 registers
constexpr int kRChunks = (kFastMaxDim / 4 + kRGT - 1) / kRGT;  // float4 chunks per consumer thread (5)
constexpr int kRChunkMax = 1024;                     // tokens sorted per chunk
constexpr int kRRingBytes = 160 * 1024;
constexpr int kRSlotsMax = 16;                       // per group
constexpr long long kRNoId = 0x7fffffffffffffffLL;   // sort key of an id outside [0, V)

// slots per group ring
__host__ __device__ constexpr int runs_slots(int dim) {
  return kRRingBytes / (kRGroups * dim * 4) < kRSlotsMax ? kRRingBytes / (kRGroups * dim * 4) : kRSlotsMax;
}
// the two rings, gamma, then the sort keys, positions and per-position statistics
__host__ __device__ constexpr int runs_smem_bytes(int dim) {
  return kRGroups * runs_slots(dim) * dim * 4 + dim * 4 + kRChunkMax * (8 + 4 + 4 + 4);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait that also gives up at once when the CTA's fail flag is set;
// a wait that runs out sets the flag and the device fault word.
__device__ __forceinline__ bool mbar_wait_or_fail(uint64_t* bar, uint32_t parity, volatile int* fail) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try(a, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 24); ++i) {
    if (mbar_try(a, parity)) return true;
    if (*fail) return false;
    if (global_ns() - t0 > 1000000000ull) break;
  }
  *fail = 1;
  atomicOr(&g_embed_fault, 1u);
  return false;
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// Named barrier of consumer group g (barrier 0 is __syncthreads).
__device__ __forceinline__ void rgroup_sync(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(g + 1), "n"(kRGT) : "memory");
}

// Next ring position: slot index and the parity of its current round.
__device__ __forceinline__ void ring_next(int& slot, uint32_t& phase, int nslots) {
  if (++slot == nslots) {
    slot = 0;
    phase ^= 1u;
  }
}

__global__ void __launch_bounds__(kRThreads, 1)
embed_bwd_runs_kernel(const int64_t* __restrict__ ids, int64_t num_tokens, const float* __restrict__ w,
                      int64_t vocab, int dim, const float* __restrict__ gamma, const float* __restrict__ mean,
                      const float* __restrict__ rstd, const float* __restrict__ dy, float* __restrict__ dw,
                      float* __restrict__ dgamma, float* __restrict__ dbeta, int chunk, int vec_gb) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int nslots = runs_slots(dim);
  float* const s_gamma = reinterpret_cast<float*>(smem_raw) + static_cast<size_t>(kRGroups) * nslots * dim;
  long long* const s_key = reinterpret_cast<long long*>(s_gamma + dim);
  int* const s_pos = reinterpret_cast<int*>(s_key + kRChunkMax);
  float* const s_mu = reinterpret_cast<float*>(s_pos + kRChunkMax);
  float* const s_rs = s_mu + kRChunkMax;
  __shared__ __align__(8) uint64_t s_full_all[kRGroups][kRSlotsMax];
  __shared__ __align__(8) uint64_t s_empty_all[kRGroups][kRSlotsMax];
  __shared__ __align__(16) float s_red[kRGroups][2][2][8];  // warp partials, entry 7 stays 0
  __shared__ int s_nvalid;
  __shared__ int s_fail_flag;
  volatile int* const s_fail = &s_fail_flag;

  const int tid = threadIdx.x, lane = tid & 31;
  const bool producer = tid >= kRCons;
  // group served (consumers: their group; producers: warp kRCons/32 + g feeds group g),
  // and a consumer's thread and warp within its group
  const int grp = producer ? (tid - kRCons) / 32 : tid / kRGT;
  const int gt = tid % kRGT, gw = gt >> 5;
  float* const ring = reinterpret_cast<float*>(smem_raw) + static_cast<size_t>(grp) * nslots * dim;
  uint64_t* const s_full = s_full_all[grp];
  uint64_t* const s_empty = s_empty_all[grp];
  const int nch = dim >> 2;
  const float fdim = static_cast<float>(dim);
  const uint32_t row_bytes = static_cast<uint32_t>(dim) * 4u;
  if (tid == 0) {
    for (int g = 0; g < kRGroups; ++g) {
      for (int i = 0; i < nslots; ++i) {
        mbar_init(&s_full_all[g][i], 1);
        mbar_init(&s_empty_all[g][i], kRGWarps);  // released by the group's warps
      }
    }
    s_fail_flag = 0;
    for (int i = 0; i < kRGroups * 2 * 2 * 8; ++i) (&s_red[0][0][0][0])[i] = 0.0f;
  }
  for (int c = tid; c < nch; c += kRThreads)
    reinterpret_cast<float4*>(s_gamma)[c] = ldg4(gamma + 4 * c);
  __syncthreads();

  // producer state (lane 0 of each producer warp)
  uint64_t evict_first = 0;
  if (producer && lane == 0) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
  uint32_t walked = 0;      // ring items walked (a failure stops the copies, not the walk)
  uint32_t used = 0, last_par = 0;  // per slot: ever filled, parity of its last fill
  // position in the group's ring, walked alike by its producer and consumers
  int slot = 0;
  uint32_t phase = 0;
  uint32_t run = 0;         // runs seen so far; run r belongs to group r & 1
  float4 S[kRChunks], pg[kRChunks], pb[kRChunks];
#pragma unroll
  for (int k = 0; k < kRChunks; ++k) S[k] = pg[k] = pb[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  int red_par = 0;

  const int64_t nchunks = (num_tokens + chunk - 1) / chunk;
  for (int64_t ch = blockIdx.x; ch < nchunks; ch += gridDim.x) {
    const int64_t c0 = ch * chunk;
    const int cnt = static_cast<int>(num_tokens - c0 < chunk ? num_tokens - c0 : chunk);
    int p2 = 1;
    while (p2 < cnt) p2 <<= 1;
    // (id, position) keys; ids outside [0, V) sort last and are left out
    for (int i = tid; i < p2; i += kRThreads) {
      long long key = kRNoId;
      if (i < cnt) {
        const int64_t id = ids[c0 + i];
        if (id >= 0 && id < vocab) key = id;
        s_mu[i] = mean[c0 + i];  // by position in the chunk, read with the ids
        s_rs[i] = rstd[c0 + i];
      }
      s_key[i] = key;
      s_pos[i] = i;
    }
    if (tid == 0) s_nvalid = 0;
    __syncthreads();
    // the pairs in ascending order of id, then position.  Up to one key per
    // thread: rank sort (each thread counts the keys before its own, reading
    // them as broadcasts; one barrier, against the bitonic network's
    // log2(p2) (log2(p2) + 1) / 2 barriers: 100.3 against 101-102 us per
    // 16,384-token backward).  Longer chunks: bitonic sort.
    if (cnt <= kRThreads) {
      long long ki = 0;
      int r = 0;
      if (tid < cnt) {
        ki = s_key[tid];
        for (int j = 0; j < cnt; ++j) {
          const long long kj = s_key[j];
          r += (kj < ki || (kj == ki && j < tid)) ? 1 : 0;
        }
      }
      __syncthreads();
      if (tid < cnt) {
        s_key[r] = ki;
        s_pos[r] = tid;
      }
      __syncthreads();
    } else {
      for (int k = 2; k <= p2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
          for (int i = tid; i < p2; i += kRThreads) {
            const int l = i ^ j;
            if (l > i) {
              const long long ki = s_key[i], kl = s_key[l];
              const int pi = s_pos[i], pl = s_pos[l];
              const bool gt2 = ki > kl || (ki == kl && pi > pl);
              if (gt2 == ((i & k) == 0)) {
                s_key[i] = kl; s_key[l] = ki;
                s_pos[i] = pl; s_pos[l] = pi;
              }
            }
          }
          __syncthreads();
        }
      }
    }
    for (int i = tid; i < p2; i += kRThreads)
      if (s_key[i] != kRNoId && (i + 1 == p2 || s_key[i + 1] == kRNoId)) s_nvalid = i + 1;
    __syncthreads();
    const int nv = s_nvalid;

    if (producer) {
      if (lane == 0) {
        auto issue = [&](const float* src, bool stream) {
          if (walked >= static_cast<uint32_t>(nslots)) mbar_wait_or_fail(&s_empty[slot], phase ^ 1u, s_fail);
          if (!*s_fail) {  // the flag never clears: after a failure no copy starts
            mbar_expect_tx(&s_full[slot], row_bytes);
            if (stream) bulk_g2s_hint(ring + static_cast<size_t>(slot) * dim, src, row_bytes, &s_full[slot], evict_first);
            else bulk_g2s(ring + static_cast<size_t>(slot) * dim, src, row_bytes, &s_full[slot]);
            used |= 1u << slot;
            last_par = (last_par & ~(1u << slot)) | (phase << slot);
          }
          ++walked;
          ring_next(slot, phase, nslots);
        };
        for (int j = 0; j < nv; ++j) {
          const bool mine = static_cast<int>(run & 1u) == grp;
          if (mine) issue(dy + (c0 + s_pos[j]) * static_cast<int64_t>(dim), true);
          if (j + 1 == nv || s_key[j + 1] != s_key[j]) {
            if (mine) issue(w + s_key[j] * static_cast<int64_t>(dim), false);
            ++run;
          }
        }
      }
    } else {
      for (int j = 0; j < nv; ++j) {
        const bool mine = static_cast<int>(run & 1u) == grp;
        if (mine) {  // a dL/dy row of this group's run: S += row
          mbar_wait_or_fail(&s_full[slot], phase, s_fail);
          const float* row = ring + static_cast<size_t>(slot) * dim;
#pragma unroll
          for (int k = 0; k < kRChunks; ++k) {
            const int c = gt + kRGT * k;
            if (c < nch) {
              const float4 d = ld4(row + 4 * c);
              const float2 lo = bwd::add2(make_float2(S[k].x, S[k].y), make_float2(d.x, d.y));
              const float2 hi = bwd::add2(make_float2(S[k].z, S[k].w), make_float2(d.z, d.w));
              S[k] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[slot]);
          ring_next(slot, phase, nslots);
        }
        if (j + 1 < nv && s_key[j + 1] == s_key[j]) continue;
        ++run;
        if (!mine) continue;  // the other group's run
        // the run's weight row: one LayerNorm backward on S
        mbar_wait_or_fail(&s_full[slot], phase, s_fail);
        const float* xs = ring + static_cast<size_t>(slot) * dim;
        const int pj = s_pos[j];
        const float r = s_rs[pj];
        const float2 r2 = bwd::dup2(r), nmu2 = bwd::dup2(-s_mu[pj]);
        // per element pair: xhat = (x - mean) r, G = S gamma, sums of G and G xhat
        float2 xh[2 * kRChunks], G[2 * kRChunks];
        float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < kRChunks; ++k) {
          const int c = gt + kRGT * k;
          if (c < nch) {
            const float4 x = ld4(xs + 4 * c);
            const float4 g4 = ld4(s_gamma + 4 * c);
            xh[2 * k] = bwd::mul2(bwd::add2(make_float2(x.x, x.y), nmu2), r2);
            xh[2 * k + 1] = bwd::mul2(bwd::add2(make_float2(x.z, x.w), nmu2), r2);
            G[2 * k] = bwd::mul2(make_float2(S[k].x, S[k].y), make_float2(g4.x, g4.y));
            G[2 * k + 1] = bwd::mul2(make_float2(S[k].z, S[k].w), make_float2(g4.z, g4.w));
            a0 = bwd::add2(a0, bwd::add2(G[2 * k], G[2 * k + 1]));
            a1 = bwd::fma2(G[2 * k], xh[2 * k], bwd::fma2(G[2 * k + 1], xh[2 * k + 1], a1));
          } else {
            xh[2 * k] = xh[2 * k + 1] = G[2 * k] = G[2 * k + 1] = make_float2(0.0f, 0.0f);
          }
        }
        float s2[2] = {__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y)};
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[slot]);
        ring_next(slot, phase, nslots);
        s2[0] = warp_sum(s2[0]);
        s2[1] = warp_sum(s2[1]);
        if (lane == 0) {
          s_red[grp][red_par][0][gw] = s2[0];
          s_red[grp][red_par][1][gw] = s2[1];
        }
        rgroup_sync(grp);
        float tot[2];
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const float4 a = *reinterpret_cast<const float4*>(&s_red[grp][red_par][v][0]);
          const float4 b = *reinterpret_cast<const float4*>(&s_red[grp][red_par][v][4]);
          tot[v] = __fadd_rn(__fadd_rn(__fadd_rn(a.x, a.y), __fadd_rn(a.z, a.w)),
                             __fadd_rn(__fadd_rn(b.x, b.y), __fadd_rn(b.z, b.w)));
        }
        red_par ^= 1;
        // dx = r (G - m1 - xhat m2) = G r + (xhat (-m2 r) - m1 r), m the row means of G and G xhat
        const float m1 = __fdiv_rn(tot[0], fdim), m2 = __fdiv_rn(tot[1], fdim);
        const float2 nm2r = bwd::dup2(-__fmul_rn(m2, r)), nm1r = bwd::dup2(-__fmul_rn(m1, r));
        float* dwrow = dw + s_key[j] * static_cast<int64_t>(dim);
#pragma unroll
        for (int k = 0; k < kRChunks; ++k) {
          const int c = gt + kRGT * k;
          if (c < nch) {
            const float2 d0 = bwd::fma2(G[2 * k], r2, bwd::fma2(xh[2 * k], nm2r, nm1r));
            const float2 d1 = bwd::fma2(G[2 * k + 1], r2, bwd::fma2(xh[2 * k + 1], nm2r, nm1r));
            red_add4(dwrow + 4 * c, make_float4(d0.x, d0.y, d1.x, d1.y));
            const float2 g0 = bwd::fma2(make_float2(S[k].x, S[k].y), xh[2 * k], make_float2(pg[k].x, pg[k].y));
            const float2 g1 = bwd::fma2(make_float2(S[k].z, S[k].w), xh[2 * k + 1], make_float2(pg[k].z, pg[k].w));
            pg[k] = make_float4(g0.x, g0.y, g1.x, g1.y);
            const float2 b0 = bwd::add2(make_float2(S[k].x, S[k].y), make_float2(pb[k].x, pb[k].y));
            const float2 b1 = bwd::add2(make_float2(S[k].z, S[k].w), make_float2(pb[k].z, pb[k].w));
            pb[k] = make_float4(b0.x, b0.y, b1.x, b1.y);
          }
          S[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
      }
    }
    __syncthreads();  // the next chunk's keys overwrite this one's
  }
  // After a failure, let the last copy issued into each slot land (bounded)
  // before the rings' shared memory is reused below.
  if (producer && lane == 0 && *s_fail) {
    for (int i = 0; i < nslots; ++i)
      if ((used >> i) & 1u) mbar_wait(&s_full[i], (last_par >> i) & 1u);
  }
  // dgamma / dbeta: group 1's partials join group 0's through shared memory
  // (the rings are idle now), then one add per column per CTA.  Every CTA
  // adds into the same 2 x D floats at about the same time, so the adds are
  // vector reductions where dgamma and dbeta are 16-byte aligned, and each
  // CTA starts at its own column so concurrent adds fall on different L2
  // lines.
  __syncthreads();
  float4* const xpg = reinterpret_cast<float4*>(smem_raw);
  float4* const xpb = xpg + nch;
  if (!producer && grp == 1) {
#pragma unroll
    for (int k = 0; k < kRChunks; ++k) {
      const int c = gt + kRGT * k;
      if (c < nch) {
        xpg[c] = pg[k];
        xpb[c] = pb[k];
      }
    }
  }
  __syncthreads();
  if (!producer && grp == 0) {
    const int rot = static_cast<int>((static_cast<int64_t>(blockIdx.x) * nch) / gridDim.x);
#pragma unroll
    for (int k = 0; k < kRChunks; ++k) {
      const int c0 = gt + kRGT * k;
      if (c0 < nch) {
        const float4 og = xpg[c0], ob = xpb[c0];
        const float4 tg = make_float4(__fadd_rn(pg[k].x, og.x), __fadd_rn(pg[k].y, og.y), __fadd_rn(pg[k].z, og.z),
                                      __fadd_rn(pg[k].w, og.w));
        const float4 tb = make_float4(__fadd_rn(pb[k].x, ob.x), __fadd_rn(pb[k].y, ob.y), __fadd_rn(pb[k].z, ob.z),
                                      __fadd_rn(pb[k].w, ob.w));
        xpg[c0] = tg;
        xpb[c0] = tb;
      }
    }
    rgroup_sync(0);
    for (int i = gt; i < nch; i += kRGT) {
      const int c = i + rot < nch ? i + rot : i + rot - nch;
      const float4 tg = xpg[c], tb = xpb[c];
      if (vec_gb) {
        red_add4(dgamma + 4 * c, tg);
        red_add4(dbeta + 4 * c, tb);
      } else {  // dgamma and dbeta need only 4-byte alignment
        atomicAdd(dgamma + 4 * c, tg.x); atomicAdd(dgamma + 4 * c + 1, tg.y);
        atomicAdd(dgamma + 4 * c + 2, tg.z); atomicAdd(dgamma + 4 * c + 3, tg.w);
        atomicAdd(dbeta + 4 * c, tb.x); atomicAdd(dbeta + 4 * c + 1, tb.y);
        atomicAdd(dbeta + 4 * c + 2, tb.z); atomicAdd(dbeta + 4 * c + 3, tb.w);
      }
    }
  }
}

// Self-test of the bounded waits: one CTA waits for the first phase of an
// mbarrier that expects one arrival nobody makes.  Every thread's wait gives
// up after about a second and the kernel sets the fault word and returns.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel() {
  __shared__ __align__(8) uint64_t s_bar;
  if (threadIdx.x == 0) mbar_init(&s_bar, 1);
  __syncthreads();
  if (!mbar_wait(&s_bar, 0u) && threadIdx.x == 0) atomicOr(&g_embed_fault, 1u);
}

// --------------------------------------------------------------------------
// host side

struct EmbedDevice {
  bool ready = false;
  unsigned long long ctx = 0;  // context the kernel attributes were set in
  int num_sms = 0;
  int occ_fwd = 1;
  int occ_slow_fwd = 1;
  int occ_slow_bwd = 1;
};

std::mutex g_mu;
EmbedDevice g_dev[kMaxDevices];

bwd_status ensure_device(EmbedDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(BWD_ERR_CUDA, "device ordinal %d unsupported", dev);
  unsigned long long ctx = 0;
  bwd_status s = bwd::host::current_context_id(&ctx);
  if (s != BWD_OK) return s;
  std::lock_guard<std::mutex> lock(g_mu);
  EmbedDevice& d = g_dev[dev];
  if (!d.ready || d.ctx != ctx) {
    d.ready = false;
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaFuncSetAttribute(reinterpret_cast<const void*>(embed_bwd_runs_kernel),
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, runs_smem_bytes(kFastMaxDim))) !=
        cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)");
    struct { const void* fn; int threads; int* out; } occ[] = {
        {reinterpret_cast<const void*>(embed_fwd_kernel), kGroup * kFwdGroups, &d.occ_fwd},
        {reinterpret_cast<const void*>(embed_fwd_slow_kernel), kGroup * kSlowGroups, &d.occ_slow_fwd},
        {reinterpret_cast<const void*>(embed_bwd_slow_kernel), kGroup * kSlowGroups, &d.occ_slow_bwd}};
    for (auto& o : occ) {
      int v = 0;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, o.fn, o.threads, 0)) != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
      *o.out = v > 0 ? v : 1;
    }
    d.ctx = ctx;
    d.ready = true;
  }
  *out = &d;
  return BWD_OK;
}

// CTAs for `tokens` tokens at `per_cta` tokens at a time: enough to cover
// them, at most one wave of resident CTAs.
int grid_for(int64_t tokens, int per_cta, int num_sms, int occ) {
  const int64_t need = (tokens + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms) * occ;
  return static_cast<int>(need < cap ? need : cap);
}

bwd_status check_shape(int64_t num_embeddings, int64_t dim) {
  if (num_embeddings < 1 || dim < 1) return fail(BWD_ERR_INVALID_ARG, "num_embeddings and dim must be >= 1");
  if (num_embeddings > INT64_MAX / dim) return fail(BWD_ERR_INVALID_ARG, "num_embeddings * dim overflows");
  return BWD_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI

extern "C" {

bwd_status bwd_embedding_init(const uint32_t* words, int64_t num_embeddings, int64_t dim, float* weight,
                              void* stream) {
  bwd_status s = check_shape(num_embeddings, dim);
  if (s != BWD_OK) return s;
  if (!words || !weight) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned_to(words, 4) || !aligned_to(weight, 4))
    return fail(BWD_ERR_INVALID_ARG, "pointer not aligned to its element size");
  EmbedDevice* d = nullptr;
  if ((s = ensure_device(&d)) != BWD_OK) return s;
  const int64_t n = num_embeddings * dim;
  const float bound = static_cast<float>(std::sqrt(6.0 / (static_cast<double>(num_embeddings) + static_cast<double>(dim))));
  const int64_t need = (n + kInitThreads - 1) / kInitThreads;
  const int64_t cap = static_cast<int64_t>(d->num_sms) * 8;
  embed_init_kernel<<<static_cast<int>(need < cap ? need : cap), kInitThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      words, n, bound, weight);
  return check_launch("embed_init_kernel launch");
}

bwd_status bwd_check_device(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int fault = 0;
  if ((e = cudaMemcpyFromSymbol(&fault, g_embed_fault, sizeof fault)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyFromSymbol(fault word)");
  if (fault == 0) return BWD_OK;
  const unsigned int zero = 0;
  if ((e = cudaMemcpyToSymbol(g_embed_fault, &zero, sizeof zero)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyToSymbol(fault word)");
  return fail(BWD_ERR_CUDA, "a bounded wait for a bulk copy in a library kernel gave up; the outputs of the "
                            "kernels since the last check are unspecified");
}

bwd_status bwd_selftest_bounded_wait(void* stream) {
  EmbedDevice* d = nullptr;
  bwd_status s = ensure_device(&d);
  if (s != BWD_OK) return s;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
  return check_launch("bounded_wait_selftest_kernel launch");
}

float bwd_embedding_xavier_bound(int64_t num_embeddings, int64_t dim) {
  if (num_embeddings < 1 || dim < 1) return -1.0f;
  return static_cast<float>(std::sqrt(6.0 / (static_cast<double>(num_embeddings) + static_cast<double>(dim))));
}

bwd_status bwd_embedding_forward(const int64_t* ids, int64_t num_tokens, const float* weight, int64_t num_embeddings,
                                 int64_t dim, const float* gamma, const float* beta, float eps, float* y,
                                 float* mean, float* rstd, void* stream) {
  bwd_status s = check_shape(num_embeddings, dim);
  if (s != BWD_OK) return s;
  if (num_tokens < 0) return fail(BWD_ERR_INVALID_ARG, "num_tokens < 0");
  if (!std::isfinite(eps) || eps < 0.0f) return fail(BWD_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (num_tokens > INT64_MAX / dim) return fail(BWD_ERR_INVALID_ARG, "num_tokens * dim overflows");
  if (num_tokens == 0) return BWD_OK;
  if (!ids || !weight || !gamma || !beta || !y) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned_to(ids, 8) || !aligned_to(weight, 4) || !aligned_to(gamma, 4) || !aligned_to(beta, 4) ||
      !aligned_to(y, 4) || !aligned_to(mean, 4) || !aligned_to(rstd, 4))
    return fail(BWD_ERR_INVALID_ARG, "pointer not aligned to its element size");
  EmbedDevice* d = nullptr;
  if ((s = ensure_device(&d)) != BWD_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool fast = dim % 4 == 0 && dim <= kFastMaxDim && aligned16(weight) && aligned16(gamma) &&
                    aligned16(beta) && aligned16(y);
  if (fast) {
    embed_fwd_kernel<<<grid_for(num_tokens, kFwdGroups, d->num_sms, d->occ_fwd), kGroup * kFwdGroups, 0, st>>>(
        ids, num_tokens, weight, num_embeddings, static_cast<int>(dim), gamma, beta, eps, y, mean, rstd);
    return check_launch("embed_fwd_kernel launch");
  }
  embed_fwd_slow_kernel<<<grid_for(num_tokens, kSlowGroups, d->num_sms, d->occ_slow_fwd), kGroup * kSlowGroups, 0,
                          st>>>(ids, num_tokens, weight, num_embeddings, dim, gamma, beta, eps, y, mean, rstd);
  return check_launch("embed_fwd_slow_kernel launch");
}

bwd_status bwd_embedding_backward(const int64_t* ids, int64_t num_tokens, const float* weight,
                                  int64_t num_embeddings, int64_t dim, const float* gamma, const float* mean,
                                  const float* rstd, const float* dy, float* dweight, float* dgamma, float* dbeta,
                                  void* stream) {
  bwd_status s = check_shape(num_embeddings, dim);
  if (s != BWD_OK) return s;
  if (num_tokens < 0) return fail(BWD_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens > INT64_MAX / dim) return fail(BWD_ERR_INVALID_ARG, "num_tokens * dim overflows");
  if (num_tokens == 0) return BWD_OK;
  if (!ids || !weight || !gamma || !mean || !rstd || !dy || !dweight || !dgamma || !dbeta)
    return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned_to(ids, 8) || !aligned_to(weight, 4) || !aligned_to(gamma, 4) || !aligned_to(mean, 4) ||
      !aligned_to(rstd, 4) || !aligned_to(dy, 4) || !aligned_to(dweight, 4) || !aligned_to(dgamma, 4) ||
      !aligned_to(dbeta, 4))
    return fail(BWD_ERR_INVALID_ARG, "pointer not aligned to its element size");
  EmbedDevice* d = nullptr;
  if ((s = ensure_device(&d)) != BWD_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool fast = dim % 4 == 0 && dim <= kFastMaxDim && aligned16(weight) && aligned16(gamma) &&
                    aligned16(dy) && aligned16(dweight);
  if (fast) {
    // one CTA per SM, each on chunks of consecutive tokens (at most 1,024)
    int64_t chunk = (num_tokens + d->num_sms - 1) / d->num_sms;
    if (chunk > kRChunkMax) chunk = kRChunkMax;
    const int64_t nchunks = (num_tokens + chunk - 1) / chunk;
    const int grid = static_cast<int>(nchunks < d->num_sms ? nchunks : d->num_sms);
    embed_bwd_runs_kernel<<<grid, kRThreads, runs_smem_bytes(static_cast<int>(dim)), st>>>(
        ids, num_tokens, weight, num_embeddings, static_cast<int>(dim), gamma, mean, rstd, dy, dweight, dgamma, dbeta,
        static_cast<int>(chunk), aligned16(dgamma) && aligned16(dbeta) ? 1 : 0);
    return check_launch("embed_bwd_runs_kernel launch");
  }
  embed_bwd_slow_kernel<<<grid_for(num_tokens, kSlowGroups, d->num_sms, d->occ_slow_bwd), kGroup * kSlowGroups, 0,
                          st>>>(ids, num_tokens, weight, num_embeddings, dim, gamma, mean, rstd, dy, dweight, dgamma,
                                dbeta);
  return check_launch("embed_bwd_slow_kernel launch");
}

}  // extern "C"
