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
// Backward, fast path: one 768-thread CTA per SM, three groups of 256
// threads.  Thread 0 of a group copies the weight row and the dy row of the
// group's NEXT token into the second of two shared-memory buffers
// (cp.async.bulk, completion counted on one mbarrier per buffer) while the
// group works on the current token from the first: xhat from the saved mean
// and rstd, the two sums of g = dy gamma and g xhat, then
// dx = rstd (g - mean(g) - xhat mean(g xhat)) added into the weight row with
// vector reductions (red.global.add.v4.f32; tokens repeat, so the adds are
// atomic).  The rows live in shared memory, not registers, so the loads of
// the next token overlap all of the current one's arithmetic; each thread
// keeps dgamma and dbeta for its own columns in registers, and each CTA adds
// the sum of its groups' partials into dgamma and dbeta once at the end
// (0.144 ms with the rows in registers and an L2 prefetch, 0.115 ms staged,
// on the 32,000 x 4,096 / 16,384-token case).  Other shapes take a
// per-element path with the same arithmetic.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "bwd.h"
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
// backward, fast path: rows staged in shared memory by bulk copies
//
// Every wait here is bounded: after about a second (or 2^24 polls) it gives
// up, sets g_embed_fault (read and cleared by bwd_check_device), and the
// group leaves its loop at the next group barrier after letting its copy in
// flight land, again with a bounded wait.
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

constexpr int kSG = 256;                 // threads per token, staged backward
constexpr int kSGWarps = kSG / 32;
constexpr int kSGroups = 3;              // groups per CTA, one CTA per SM
constexpr int kSChunks = kFastMaxDim / (4 * kSG);  // 4 float4 chunks per thread

__host__ __device__ constexpr int staged_smem_bytes(int dim) { return kSGroups * 2 * 2 * dim * 4; }

__device__ __forceinline__ void group_sync256(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "n"(kSG) : "memory");
}

template <int kVals>
__device__ __forceinline__ void group_sum256(float (&v)[kVals], float* red, int slot, int group, int t) {
  const int lane = t & 31, warp = t >> 5;
#pragma unroll
  for (int i = 0; i < kVals; ++i) v[i] = warp_sum(v[i]);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kVals; ++i) red[(slot * kVals + i) * kSGWarps + warp] = v[i];
  }
  group_sync256(group);
#pragma unroll
  for (int i = 0; i < kVals; ++i) {
    const float4 a = *reinterpret_cast<const float4*>(&red[(slot * kVals + i) * kSGWarps]);
    const float4 b = *reinterpret_cast<const float4*>(&red[(slot * kVals + i) * kSGWarps + 4]);
    v[i] = __fadd_rn(__fadd_rn(__fadd_rn(a.x, a.y), __fadd_rn(a.z, a.w)), __fadd_rn(__fadd_rn(b.x, b.y), __fadd_rn(b.z, b.w)));
  }
}

// Backward with the rows staged in shared memory: thread 0 of each group
// copies the next token's weight and dy rows (cp.async.bulk, one mbarrier
// per buffer) while the group works on the current token from the other
// buffer; dgamma / dbeta partials stay in registers.
__global__ void __launch_bounds__(kSG * kSGroups, 1)
embed_bwd_staged_kernel(const int64_t* __restrict__ ids, int64_t num_tokens, const float* __restrict__ w, int64_t vocab,
                        int dim, const float* __restrict__ gamma, const float* __restrict__ mean,
                        const float* __restrict__ rstd, const float* __restrict__ dy, float* __restrict__ dw,
                        float* __restrict__ dgamma, float* __restrict__ dbeta) {
  extern __shared__ __align__(128) float s_buf[];  // [group][buffer][x | dy][dim]
  __shared__ __align__(16) float s_red[kSGroups][2 * 2 * kSGWarps];
  __shared__ __align__(8) uint64_t s_full[kSGroups][2];
  // s_abort[group][c]: a wait gave up in an iteration of parity 1 - c.  All
  // threads read cell (it & 1) right after the loop-top barrier of
  // iteration it.  Writes to that cell come from iteration it - 1, finished
  // before that barrier, or from iteration it + 1, which no thread enters
  // before every thread has reached the next loop-top barrier, after its
  // read: so all threads of the group decide alike.
  __shared__ int s_abort[kSGroups][2];
  const int group = threadIdx.x / kSG, t = threadIdx.x % kSG;
  const int nch = dim >> 2;
  const float fdim = static_cast<float>(dim);
  const uint32_t row_bytes = static_cast<uint32_t>(dim) * 4u;
  float* const gbuf = s_buf + static_cast<int64_t>(group) * 4 * dim;
  if (t == 0) {
    mbar_init(&s_full[group][0], 1);
    mbar_init(&s_full[group][1], 1);
    s_abort[group][0] = s_abort[group][1] = 0;
  }
  __syncthreads();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kSGroups;
  const int64_t tok0 = static_cast<int64_t>(blockIdx.x) * kSGroups + group;
  // copies of token `tok` into buffer `b` (nothing for an id outside [0, V));
  // thread 0 counts the phases it started per buffer (for the drain below)
  uint32_t issued[2] = {0u, 0u};
  auto issue = [&](int64_t tok, int b) {
    const int64_t id = ids[tok];
    if (id < 0 || id >= vocab) return;
    ++issued[b];
    uint64_t* bar = &s_full[group][b];
    mbar_expect_tx(bar, 2u * row_bytes);
    bulk_g2s(gbuf + b * 2 * dim, w + id * static_cast<int64_t>(dim), row_bytes, bar);
    bulk_g2s(gbuf + b * 2 * dim + dim, dy + tok * static_cast<int64_t>(dim), row_bytes, bar);
  };
  if (t == 0 && tok0 < num_tokens) issue(tok0, 0);
  float4 pg[kSChunks], pb[kSChunks];
#pragma unroll
  for (int k = 0; k < kSChunks; ++k) pg[k] = pb[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  uint32_t phase = 0;  // bit b: parity of buffer b's next phase
  int slot = 0;
  int it = 0;
  for (int64_t tok = tok0; tok < num_tokens; tok += stride, ++it) {
    const int b = it & 1;
    group_sync256(group);  // every thread is done with the other buffer
    if (s_abort[group][it & 1]) break;
    if (t == 0 && tok + stride < num_tokens) issue(tok + stride, b ^ 1);
    const int64_t id = ids[tok];
    if (id < 0 || id >= vocab) continue;  // the whole group skips together
    const bool ok = mbar_wait(&s_full[group][b], (phase >> b) & 1u);
    phase ^= 1u << b;
    if (!ok) {
      atomicOr(&g_embed_fault, 1u);
      s_abort[group][(it + 1) & 1] = 1;
    }
    const float mu = mean[tok], r = rstd[tok];
    const float* xs = gbuf + b * 2 * dim;
    const float* ds = xs + dim;
    float s[2] = {0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < kSChunks; ++k) {
      const int c = t + kSG * k;
      if (c < nch) {
        const float4 x = *reinterpret_cast<const float4*>(xs + 4 * c);
        const float4 d = *reinterpret_cast<const float4*>(ds + 4 * c);
        const float4 g = ldg4(gamma + 4 * c);
        const float4 xh = make_float4(__fmul_rn(__fsub_rn(x.x, mu), r), __fmul_rn(__fsub_rn(x.y, mu), r),
                                      __fmul_rn(__fsub_rn(x.z, mu), r), __fmul_rn(__fsub_rn(x.w, mu), r));
        const float4 gg = make_float4(__fmul_rn(d.x, g.x), __fmul_rn(d.y, g.y), __fmul_rn(d.z, g.z), __fmul_rn(d.w, g.w));
        s[0] = __fadd_rn(s[0], __fadd_rn(__fadd_rn(gg.x, gg.y), __fadd_rn(gg.z, gg.w)));
        s[1] = __fadd_rn(s[1], __fadd_rn(__fadd_rn(__fmul_rn(gg.x, xh.x), __fmul_rn(gg.y, xh.y)),
                                         __fadd_rn(__fmul_rn(gg.z, xh.z), __fmul_rn(gg.w, xh.w))));
        if (ok) {
          pg[k].x = __fadd_rn(pg[k].x, __fmul_rn(d.x, xh.x));
          pg[k].y = __fadd_rn(pg[k].y, __fmul_rn(d.y, xh.y));
          pg[k].z = __fadd_rn(pg[k].z, __fmul_rn(d.z, xh.z));
          pg[k].w = __fadd_rn(pg[k].w, __fmul_rn(d.w, xh.w));
          pb[k].x = __fadd_rn(pb[k].x, d.x);
          pb[k].y = __fadd_rn(pb[k].y, d.y);
          pb[k].z = __fadd_rn(pb[k].z, d.z);
          pb[k].w = __fadd_rn(pb[k].w, d.w);
        }
      }
    }
    group_sum256<2>(s, s_red[group], slot, group, t);
    slot ^= 1;
    const float m1 = __fdiv_rn(s[0], fdim), m2 = __fdiv_rn(s[1], fdim);
    float* dwrow = dw + id * static_cast<int64_t>(dim);
#pragma unroll
    for (int k = 0; k < kSChunks; ++k) {
      const int c = t + kSG * k;
      if (c < nch && ok) {
        const float4 x = *reinterpret_cast<const float4*>(xs + 4 * c);
        const float4 d = *reinterpret_cast<const float4*>(ds + 4 * c);
        const float4 g = ldg4(gamma + 4 * c);
        float4 dx;
        dx.x = __fmul_rn(r, __fsub_rn(__fsub_rn(__fmul_rn(d.x, g.x), m1), __fmul_rn(__fmul_rn(__fsub_rn(x.x, mu), r), m2)));
        dx.y = __fmul_rn(r, __fsub_rn(__fsub_rn(__fmul_rn(d.y, g.y), m1), __fmul_rn(__fmul_rn(__fsub_rn(x.y, mu), r), m2)));
        dx.z = __fmul_rn(r, __fsub_rn(__fsub_rn(__fmul_rn(d.z, g.z), m1), __fmul_rn(__fmul_rn(__fsub_rn(x.z, mu), r), m2)));
        dx.w = __fmul_rn(r, __fsub_rn(__fsub_rn(__fmul_rn(d.w, g.w), m1), __fmul_rn(__fmul_rn(__fsub_rn(x.w, mu), r), m2)));
        red_add4(dwrow + 4 * c, dx);
      }
    }
  }
  // A group that gave up lets every copy it started land (bounded) before
  // the buffers are reused below: the one whose wait timed out and the one
  // issued ahead.  The k-th copy into a buffer completes its phase k - 1;
  // waiting on the parity of a phase that already completed returns at once.
  if (t == 0 && (s_abort[group][0] || s_abort[group][1])) {
#pragma unroll
    for (int b = 0; b < 2; ++b)
      if (issued[b] > 0) mbar_wait(&s_full[group][b], (issued[b] - 1u) & 1u);
  }
  __syncthreads();
  // partials: each group's into its first buffer, then summed over the groups in order
  float* const part = s_buf + static_cast<int64_t>(group) * 4 * dim;
#pragma unroll
  for (int k = 0; k < kSChunks; ++k) {
    const int c = t + kSG * k;
    if (c < nch) {
      *reinterpret_cast<float4*>(part + 4 * c) = pg[k];
      *reinterpret_cast<float4*>(part + dim + 4 * c) = pb[k];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < dim; i += blockDim.x) {
    float a = 0.0f, bsum = 0.0f;
#pragma unroll
    for (int gi = 0; gi < kSGroups; ++gi) {
      a = __fadd_rn(a, s_buf[static_cast<int64_t>(gi) * 4 * dim + i]);
      bsum = __fadd_rn(bsum, s_buf[static_cast<int64_t>(gi) * 4 * dim + dim + i]);
    }
    atomicAdd(dgamma + i, a);
    atomicAdd(dbeta + i, bsum);
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
    if ((e = cudaFuncSetAttribute(reinterpret_cast<const void*>(embed_bwd_staged_kernel),
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, staged_smem_bytes(kFastMaxDim))) !=
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
    embed_bwd_staged_kernel<<<grid_for(num_tokens, kSGroups, d->num_sms, 1), kSG * kSGroups,
                              staged_smem_bytes(static_cast<int>(dim)), st>>>(
        ids, num_tokens, weight, num_embeddings, static_cast<int>(dim), gamma, mean, rstd, dy, dweight, dgamma, dbeta);
    return check_launch("embed_bwd_staged_kernel launch");
  }
  embed_bwd_slow_kernel<<<grid_for(num_tokens, kSlowGroups, d->num_sms, d->occ_slow_bwd), kGroup * kSlowGroups, 0,
                          st>>>(ids, num_tokens, weight, num_embeddings, dim, gamma, mean, rstd, dy, dweight, dgamma,
                                dbeta);
  return check_launch("embed_bwd_slow_kernel launch");
}

}  // extern "C"
