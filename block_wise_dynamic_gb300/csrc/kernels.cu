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
// Work decomposition.  One CTA of 256 threads owns one 2048-element block at
// a time and walks blocks with a grid stride (grid = SMs x resident CTAs).
// Thread `tid` owns elements {4 tid .. 4 tid + 3} and {1024 + 4 tid .. +3} of
// the block, so every warp-wide load or store touches one contiguous span
// (512 B of fp32, 256 B of bf16, 128 B of codes) and is fully coalesced.  The
// block absmax is a warp shuffle reduction followed by a shared-memory pass
// over the 8 warps.  The map, thresholds and bucket tables live in shared
// memory.  All arithmetic that decides a code (absmax, x / absmax, the
// threshold compare) is plain IEEE binary32, with explicit round-to-nearest
// intrinsics so that no multiply-add is ever contracted.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "bwd.h"
#include "tables.h"

namespace {

using bwd::kBktBase;
using bwd::kBktPad;
using bwd::kCodes;
using bwd::kNumBkt;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTensors = 448;  // per launch, bounded by kernel parameter space
constexpr int kMaxDevices = 64;

__device__ bwd::Tables g_tables;  // immutable after the first upload per device

// --------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Number of thresholds <= y for y >= +0 given as its bit pattern (see the
// bucket table description in tables.h).  Indices are clamped, so any input
// pattern stays inside the tables.
__device__ __forceinline__ uint32_t count_le(uint32_t ybits, const uint8_t* bkt, const float* thr) {
  int b = static_cast<int>(ybits >> bwd::kBktShift) - kBktBase;
  b = min(max(b, 0), kNumBkt - 1);
  const uint32_t c = bkt[b];
  return c + (thr[c] <= __uint_as_float(ybits) ? 1u : 0u);
}

// Signed map.  For xn >= 0 (including -0.0) the code is count(xn).  The
// thresholds are antisymmetric, t[254 - i] = -t[i], so for xn = -a < 0 the
// count of thresholds <= -a is 255 - #{t < a} = 255 - count(pred(a)), where
// pred(a) is the next binary32 value below a.
__device__ __forceinline__ uint32_t code_signed(float xn, const uint8_t* bkt, const float* thr) {
  const uint32_t u = __float_as_uint(xn);
  const uint32_t a = u & 0x7fffffffu;
  const bool neg = (u != a) && (a != 0u);
  const uint32_t c = count_le(neg ? a - 1u : a, bkt, thr);
  return neg ? 255u - c : c;
}

// Unsigned map: every threshold is positive, so a negative input has code 0.
__device__ __forceinline__ uint32_t code_unsigned(float xn, const uint8_t* bkt, const float* thr) {
  const uint32_t u = __float_as_uint(xn);
  const uint32_t c = count_le(u, bkt, thr);
  return (u >> 31) ? 0u : c;
}

template <bool kSigned>
__device__ __forceinline__ uint32_t quantize_one(float x, float absmax, const uint8_t* bkt,
                                                 const float* thr) {
  const float xn = __fdiv_rn(x, absmax);
  return kSigned ? code_signed(xn, bkt, thr) : code_unsigned(xn, bkt, thr);
}

// Elements of a block present in a tensor of n elements (1..2048).
__device__ __forceinline__ int64_t rem_in_block(int64_t n, int64_t base) {
  const int64_t r = n - base;
  return r < BWD_BLOCK ? r : BWD_BLOCK;
}

// Element slot k (0..7) of thread tid inside a block.
__device__ __forceinline__ int slot_index(int tid, int k) {
  return (k < 4) ? 4 * tid + k : 1024 + 4 * tid + (k - 4);
}

__device__ __forceinline__ void copy_to_smem(void* dst, const void* src, int bytes) {
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = static_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x) d[i] = s[i];
}

// --------------------------------------------------------------------------
// quantize

template <bool kSigned>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ codes,
                float* __restrict__ absmax, int vec_ok) {
  __shared__ __align__(16) float s_thr[kCodes];
  __shared__ __align__(16) uint8_t s_bkt[kBktPad];
  __shared__ float s_red[2][kWarps];
  const int k = kSigned ? 0 : 1;
  copy_to_smem(s_thr, g_tables.thr[k], sizeof(s_thr));
  copy_to_smem(s_bkt, g_tables.bkt[k], sizeof(s_bkt));
  __syncthreads();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nb = (n + BWD_BLOCK - 1) / BWD_BLOCK;
  const uint32_t zc = kSigned ? 128u : 0u;
  int it = 0;
  for (int64_t b = blockIdx.x; b < nb; b += gridDim.x, ++it) {
    const int64_t base = b * BWD_BLOCK;
    const int rem = static_cast<int>(rem_in_block(n, base));
    const bool vec = vec_ok && rem == BWD_BLOCK;
    float v[8];
    if (vec) {
      const float4 a0 = __ldcs(reinterpret_cast<const float4*>(x + base) + tid);
      const float4 a1 = __ldcs(reinterpret_cast<const float4*>(x + base + 1024) + tid);
      v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
      v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = slot_index(tid, j);
        v[j] = e < rem ? x[base + e] : 0.0f;
      }
    }
    float mx = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(v[j]));
    mx = warp_max(mx);
    if (lane == 0) s_red[it & 1][warp] = mx;
    __syncthreads();
    float am = s_red[it & 1][0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) am = fmaxf(am, s_red[it & 1][w]);

    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      c[j] = (am == 0.0f) ? zc : quantize_one<kSigned>(v[j], am, s_bkt, s_thr);
    if (vec) {
      const uint32_t w0 = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
      const uint32_t w1 = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
      __stcs(reinterpret_cast<unsigned int*>(codes + base) + tid, w0);
      __stcs(reinterpret_cast<unsigned int*>(codes + base + 1024) + tid, w1);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = slot_index(tid, j);
        if (e < rem) codes[base + e] = static_cast<uint8_t>(c[j]);
      }
    }
    if (tid == 0) absmax[b] = am;
  }
}

// --------------------------------------------------------------------------
// dequantize

template <bool kSigned>
__global__ void __launch_bounds__(kThreads)
dequantize_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ absmax, int64_t n,
                  float* __restrict__ y, int vec_ok) {
  __shared__ __align__(16) float s_map[kCodes];
  copy_to_smem(s_map, g_tables.map[kSigned ? 0 : 1], sizeof(s_map));
  __syncthreads();
  const int tid = threadIdx.x;
  const int64_t nb = (n + BWD_BLOCK - 1) / BWD_BLOCK;
  for (int64_t b = blockIdx.x; b < nb; b += gridDim.x) {
    const int64_t base = b * BWD_BLOCK;
    const int rem = static_cast<int>(rem_in_block(n, base));
    const float am = absmax[b];
    if (vec_ok && rem == BWD_BLOCK) {
      const uint32_t w0 = __ldcs(reinterpret_cast<const unsigned int*>(codes + base) + tid);
      const uint32_t w1 = __ldcs(reinterpret_cast<const unsigned int*>(codes + base + 1024) + tid);
      float4 o0, o1;
      o0.x = __fmul_rn(s_map[w0 & 0xff], am);
      o0.y = __fmul_rn(s_map[(w0 >> 8) & 0xff], am);
      o0.z = __fmul_rn(s_map[(w0 >> 16) & 0xff], am);
      o0.w = __fmul_rn(s_map[w0 >> 24], am);
      o1.x = __fmul_rn(s_map[w1 & 0xff], am);
      o1.y = __fmul_rn(s_map[(w1 >> 8) & 0xff], am);
      o1.z = __fmul_rn(s_map[(w1 >> 16) & 0xff], am);
      o1.w = __fmul_rn(s_map[w1 >> 24], am);
      __stcs(reinterpret_cast<float4*>(y + base) + tid, o0);
      __stcs(reinterpret_cast<float4*>(y + base + 1024) + tid, o1);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = slot_index(tid, j);
        if (e < rem) y[base + e] = __fmul_rn(s_map[codes[base + e]], am);
      }
    }
  }
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
  float* p;
  const void* g;
  uint8_t* mc;
  float* ma;
  uint8_t* vc;
  float* va;
  int64_t n;
  int64_t vec;  // all six pointers 16-byte aligned
};

struct AdamArgs {
  int64_t block_start[kMaxTensors + 1];  // prefix sums of per-tensor block counts
  TensorArgs t[kMaxTensors];
  int32_t num_tensors;
  float b1, omb1, b2, omb2, eps, step_size, bc2s;
};

static_assert(sizeof(AdamArgs) <= 32764, "kernel parameter space");

template <bool kBf16>
__device__ __forceinline__ void load_grad_vec(const void* g, int64_t base, int tid, float* out) {
  if (kBf16) {
    const uint2 a0 = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(g) + base) + tid);
    const uint2 a1 =
        __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(g) + base + 1024) + tid);
    out[0] = __uint_as_float(a0.x << 16);
    out[1] = __uint_as_float(a0.x & 0xffff0000u);
    out[2] = __uint_as_float(a0.y << 16);
    out[3] = __uint_as_float(a0.y & 0xffff0000u);
    out[4] = __uint_as_float(a1.x << 16);
    out[5] = __uint_as_float(a1.x & 0xffff0000u);
    out[6] = __uint_as_float(a1.y << 16);
    out[7] = __uint_as_float(a1.y & 0xffff0000u);
  } else {
    const float4 a0 = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(g) + base) + tid);
    const float4 a1 =
        __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(g) + base + 1024) + tid);
    out[0] = a0.x; out[1] = a0.y; out[2] = a0.z; out[3] = a0.w;
    out[4] = a1.x; out[5] = a1.y; out[6] = a1.z; out[7] = a1.w;
  }
}

template <bool kBf16>
__device__ __forceinline__ float load_grad_one(const void* g, int64_t i) {
  if (kBf16) return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(g)[i]) << 16);
  return static_cast<const float*>(g)[i];
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
adam8bit_kernel(const __grid_constant__ AdamArgs args) {
  __shared__ __align__(16) bwd::Tables s_tab;
  __shared__ float s_red[2][2][kWarps];
  copy_to_smem(&s_tab, &g_tables, sizeof(bwd::Tables));
  __syncthreads();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = args.num_tensors;
  const int64_t total = args.block_start[nt];
  const int64_t first = blockIdx.x;
  if (first >= total) return;

  // tensor holding global block `first`: the last ti with block_start[ti] <= first
  int lo = 0, hi = nt - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (args.block_start[mid] <= first) lo = mid; else hi = mid - 1;
  }
  int ti = lo;

  const float b1 = args.b1, omb1 = args.omb1, b2 = args.b2, omb2 = args.omb2;
  const float eps = args.eps, step_size = args.step_size, bc2s = args.bc2s;
  int it = 0;
  for (int64_t gb = first; gb < total; gb += gridDim.x, ++it) {
    while (args.block_start[ti + 1] <= gb) ++ti;
    const TensorArgs& T = args.t[ti];
    const int64_t lb = gb - args.block_start[ti];
    const int64_t base = lb * BWD_BLOCK;
    const int rem = static_cast<int>(rem_in_block(T.n, base));
    const bool vec = T.vec && rem == BWD_BLOCK;
    const float ma_old = T.ma[lb];
    const float va_old = T.va[lb];

    float p[8], g[8];
    uint32_t mcode[8], vcode[8];
    if (vec) {
      const float4 p0 = __ldcs(reinterpret_cast<const float4*>(T.p + base) + tid);
      const float4 p1 = __ldcs(reinterpret_cast<const float4*>(T.p + base + 1024) + tid);
      p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w;
      p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
      load_grad_vec<kBf16>(T.g, base, tid, g);
      const uint32_t m0 = __ldcs(reinterpret_cast<const unsigned int*>(T.mc + base) + tid);
      const uint32_t m1 = __ldcs(reinterpret_cast<const unsigned int*>(T.mc + base + 1024) + tid);
      const uint32_t v0 = __ldcs(reinterpret_cast<const unsigned int*>(T.vc + base) + tid);
      const uint32_t v1 = __ldcs(reinterpret_cast<const unsigned int*>(T.vc + base + 1024) + tid);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mcode[j] = (m0 >> (8 * j)) & 0xffu;
        mcode[4 + j] = (m1 >> (8 * j)) & 0xffu;
        vcode[j] = (v0 >> (8 * j)) & 0xffu;
        vcode[4 + j] = (v1 >> (8 * j)) & 0xffu;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = slot_index(tid, j);
        const bool in = e < rem;
        p[j] = in ? T.p[base + e] : 0.0f;
        g[j] = in ? load_grad_one<kBf16>(T.g, base + e) : 0.0f;
        mcode[j] = in ? T.mc[base + e] : 128u;  // padding: code of +0.0
        vcode[j] = in ? T.vc[base + e] : 0u;
      }
    }

    // dequantize -> Adam in fp32 (operation order fixed, one rounding each)
    float m[8], v[8];
    float mmax = 0.0f, vmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float m_old = __fmul_rn(s_tab.map[0][mcode[j]], ma_old);
      const float v_old = __fmul_rn(s_tab.map[1][vcode[j]], va_old);
      const float gj = g[j];
      m[j] = __fadd_rn(__fmul_rn(b1, m_old), __fmul_rn(omb1, gj));
      v[j] = __fadd_rn(__fmul_rn(b2, v_old), __fmul_rn(__fmul_rn(omb2, gj), gj));
      const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v[j]), bc2s), eps);
      p[j] = __fsub_rn(p[j], __fdiv_rn(__fmul_rn(step_size, m[j]), denom));
      mmax = fmaxf(mmax, fabsf(m[j]));
      vmax = fmaxf(vmax, fabsf(v[j]));
    }
    // padding slots of a partial block (g = 0, codes of zero) give m = v = 0,
    // so they leave the block absmax unchanged

    // block absmax of the new moments
    mmax = warp_max(mmax);
    vmax = warp_max(vmax);
    if (lane == 0) { s_red[it & 1][0][warp] = mmax; s_red[it & 1][1][warp] = vmax; }
    __syncthreads();
    float am = s_red[it & 1][0][0], av = s_red[it & 1][1][0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      am = fmaxf(am, s_red[it & 1][0][w]);
      av = fmaxf(av, s_red[it & 1][1][w]);
    }

    // requantize
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      mcode[j] = (am == 0.0f) ? 128u : quantize_one<true>(m[j], am, s_tab.bkt[0], s_tab.thr[0]);
      vcode[j] = (av == 0.0f) ? 0u : quantize_one<false>(v[j], av, s_tab.bkt[1], s_tab.thr[1]);
    }

    if (vec) {
      __stcs(reinterpret_cast<float4*>(T.p + base) + tid, make_float4(p[0], p[1], p[2], p[3]));
      __stcs(reinterpret_cast<float4*>(T.p + base + 1024) + tid, make_float4(p[4], p[5], p[6], p[7]));
      __stcs(reinterpret_cast<unsigned int*>(T.mc + base) + tid,
             mcode[0] | (mcode[1] << 8) | (mcode[2] << 16) | (mcode[3] << 24));
      __stcs(reinterpret_cast<unsigned int*>(T.mc + base + 1024) + tid,
             mcode[4] | (mcode[5] << 8) | (mcode[6] << 16) | (mcode[7] << 24));
      __stcs(reinterpret_cast<unsigned int*>(T.vc + base) + tid,
             vcode[0] | (vcode[1] << 8) | (vcode[2] << 16) | (vcode[3] << 24));
      __stcs(reinterpret_cast<unsigned int*>(T.vc + base + 1024) + tid,
             vcode[4] | (vcode[5] << 8) | (vcode[6] << 16) | (vcode[7] << 24));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = slot_index(tid, j);
        if (e < rem) {
          T.p[base + e] = p[j];
          T.mc[base + e] = static_cast<uint8_t>(mcode[j]);
          T.vc[base + e] = static_cast<uint8_t>(vcode[j]);
        }
      }
    }
    // every thread read the old absmax before the barrier above
    if (tid == 0) { T.ma[lb] = am; T.va[lb] = av; }
  }
}

// --------------------------------------------------------------------------
// host side

thread_local std::string t_last_error;

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

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int occ_quant[2] = {0, 0};
  int occ_dequant[2] = {0, 0};
  int occ_adam[2] = {0, 0};
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
bwd::Tables g_host_tables;
bool g_host_built = false;

bwd_status occupancy(const void* fn, int* out) {
  int v = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, kThreads, 0);
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
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.ready) { *out = &d; return BWD_OK; }
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
  bwd_status s;
  if ((s = occupancy(reinterpret_cast<const void*>(quantize_kernel<true>), &d.occ_quant[0])) != BWD_OK) return s;
  if ((s = occupancy(reinterpret_cast<const void*>(quantize_kernel<false>), &d.occ_quant[1])) != BWD_OK) return s;
  if ((s = occupancy(reinterpret_cast<const void*>(dequantize_kernel<true>), &d.occ_dequant[0])) != BWD_OK) return s;
  if ((s = occupancy(reinterpret_cast<const void*>(dequantize_kernel<false>), &d.occ_dequant[1])) != BWD_OK) return s;
  if ((s = occupancy(reinterpret_cast<const void*>(adam8bit_kernel<false>), &d.occ_adam[0])) != BWD_OK) return s;
  if ((s = occupancy(reinterpret_cast<const void*>(adam8bit_kernel<true>), &d.occ_adam[1])) != BWD_OK) return s;
  d.ready = true;
  *out = &d;
  return BWD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int grid_for(int64_t blocks, const DeviceState& d, int occ) {
  const int64_t cap = static_cast<int64_t>(d.num_sms) * occ;
  return static_cast<int>(blocks < cap ? blocks : cap);
}

bwd_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, what);
  return BWD_OK;
}

bool valid_kind(bwd_map_kind k) { return k == BWD_MAP_SIGNED || k == BWD_MAP_UNSIGNED; }

bwd_status check_hparams(const bwd_adam_hparams* hp) {
  if (!hp) return fail(BWD_ERR_INVALID_ARG, "hparams is NULL");
  if (hp->step < 1) return fail(BWD_ERR_INVALID_ARG, "step must be >= 1 (got %lld)", (long long)hp->step);
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->eps) || hp->eps < 0.0f)
    return fail(BWD_ERR_INVALID_ARG, "lr and eps must be finite, eps >= 0");
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return fail(BWD_ERR_INVALID_ARG, "betas must lie in [0, 1)");
  if (hp->weight_decay != 0.0f) return fail(BWD_ERR_INVALID_ARG, "weight_decay must be 0");
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
  a->bc2s = static_cast<float>(std::sqrt(bc2));
}

bwd_status launch_adam_chunk(const AdamArgs& a, bool bf16, const DeviceState& d, cudaStream_t st) {
  const int64_t total = a.block_start[a.num_tensors];
  if (total == 0) return BWD_OK;
  const int grid = grid_for(total, d, d.occ_adam[bf16 ? 1 : 0]);
  if (bf16) adam8bit_kernel<true><<<grid, kThreads, 0, st>>>(a);
  else adam8bit_kernel<false><<<grid, kThreads, 0, st>>>(a);
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

const char* bwd_last_error(void) { return t_last_error.c_str(); }

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
  DeviceState* d = nullptr;
  bwd_status s = ensure_device(&d);
  if (s != BWD_OK) return s;
  const int64_t nb = bwd_num_blocks(n);
  const int vec = aligned16(x) && aligned16(codes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kind == BWD_MAP_SIGNED)
    quantize_kernel<true><<<grid_for(nb, *d, d->occ_quant[0]), kThreads, 0, st>>>(x, n, codes, absmax, vec);
  else
    quantize_kernel<false><<<grid_for(nb, *d, d->occ_quant[1]), kThreads, 0, st>>>(x, n, codes, absmax, vec);
  return check_launch("quantize_kernel launch");
}

bwd_status bwd_dequantize_blockwise(const uint8_t* codes, const float* absmax, int64_t n,
                                    bwd_map_kind kind, float* y, void* stream) {
  if (n < 0) return fail(BWD_ERR_INVALID_ARG, "n < 0");
  if (!valid_kind(kind)) return fail(BWD_ERR_INVALID_ARG, "bad map kind %d", (int)kind);
  if (n == 0) return BWD_OK;
  if (!codes || !absmax || !y) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  DeviceState* d = nullptr;
  bwd_status s = ensure_device(&d);
  if (s != BWD_OK) return s;
  const int64_t nb = bwd_num_blocks(n);
  const int vec = aligned16(codes) && aligned16(y);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kind == BWD_MAP_SIGNED)
    dequantize_kernel<true><<<grid_for(nb, *d, d->occ_dequant[0]), kThreads, 0, st>>>(codes, absmax, n, y, vec);
  else
    dequantize_kernel<false><<<grid_for(nb, *d, d->occ_dequant[1]), kThreads, 0, st>>>(codes, absmax, n, y, vec);
  return check_launch("dequantize_kernel launch");
}

bwd_status bwd_state_init(uint8_t* m_codes, float* m_absmax, uint8_t* v_codes, float* v_absmax,
                          int64_t n, void* stream) {
  if (n < 0) return fail(BWD_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return BWD_OK;
  if (!m_codes || !m_absmax || !v_codes || !v_absmax) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  DeviceState* d = nullptr;
  bwd_status s = ensure_device(&d);
  if (s != BWD_OK) return s;
  const int64_t work = (n + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(work < d->num_sms * 8 ? work : d->num_sms * 8);
  fill_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      m_codes, 128, v_codes, 0, n, m_absmax, v_absmax, bwd_num_blocks(n));
  return check_launch("fill_kernel launch");
}

bwd_status bwd_adam8bit_step_multi(int32_t num_tensors, float* const* p, const void* const* g,
                                   bwd_dtype g_dtype, uint8_t* const* m_codes, float* const* m_absmax,
                                   uint8_t* const* v_codes, float* const* v_absmax, const int64_t* n,
                                   const bwd_adam_hparams* hp, void* stream) {
  if (num_tensors < 0) return fail(BWD_ERR_INVALID_ARG, "num_tensors < 0");
  if (g_dtype != BWD_F32 && g_dtype != BWD_BF16)
    return fail(BWD_ERR_UNSUPPORTED_DTYPE, "gradient dtype %d", (int)g_dtype);
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
    any_work = any_work || n[i] > 0;
  }
  if (!any_work) return BWD_OK;
  DeviceState* d = nullptr;
  if ((s = ensure_device(&d)) != BWD_OK) return s;

  static thread_local AdamArgs a;  // ~32 KB: kept off the stack
  fill_scalars(hp, &a);
  const bool bf16 = g_dtype == BWD_BF16;
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
      if ((s = launch_adam_chunk(a, bf16, *d, st)) != BWD_OK) return s;
      k = 0;
      a.block_start[0] = 0;
    }
  }
  if (k > 0) {
    a.num_tensors = k;
    if ((s = launch_adam_chunk(a, bf16, *d, st)) != BWD_OK) return s;
  }
  return BWD_OK;
}

bwd_status bwd_adam8bit_step(float* p, const void* g, bwd_dtype g_dtype, uint8_t* m_codes,
                             float* m_absmax, uint8_t* v_codes, float* v_absmax, int64_t n,
                             const bwd_adam_hparams* hp, void* stream) {
  return bwd_adam8bit_step_multi(1, &p, &g, g_dtype, &m_codes, &m_absmax, &v_codes, &v_absmax, &n, hp,
                                 stream);
}

}  // extern "C"
