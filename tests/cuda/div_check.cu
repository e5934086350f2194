// Check of bwd::div_fast, the packed bwd::div_fast2 and the unscaled forms
// bwd::div_unscaled / div_unscaled2 (exact_div.cuh) against __fdiv_rn, bit
// for bit.
// Usage: div_check [divisor_significands [first]]; all 2^23 divisor
// significands (about 90 s on one GB300) make the check exhaustive over every
// pair of binary32 significands and both signs of the dividend.
// Part 1: every x significand in [1,2) x every divisor significand in [1,2).
// Part 2: random (x, a) over many exponents with |x/a| >= 2^-64 (and a in the
//   fast range); for the unscaled forms also |x/a| < 2^-64, where the result
//   must stay below 2^-63 in magnitude and RN(x Y) below 2^-62.
// Part 3: the unscaled forms at the ends of their divisor range (exponent
//   fields 89 and 252) with quotients around 2^-64: every x significand x the
//   same divisor significands as part 1, both signs.
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include "exact_div.cuh"

__device__ unsigned long long g_bad;
__device__ unsigned long long g_checked;
__device__ uint32_t g_first[64];  // pairs (x bits, a bits)
__device__ uint32_t g_nfirst;

__device__ void record(float x, float a) {
  uint32_t k = atomicAdd(&g_nfirst, 1u);
  if (k < 32) { g_first[2 * k] = __float_as_uint(x); g_first[2 * k + 1] = __float_as_uint(a); }
}

// grid: x dimension strides over x significands, y over divisor significands in [a_lo, a_lo + gridDim.y)
__global__ void part1(uint32_t a_lo) {
  const uint32_t ai = a_lo + blockIdx.y;
  if (ai >= (1u << 23)) return;
  const float a = __uint_as_float(0x3f800000u | ai);
  const bwd::Divisor d = bwd::make_divisor(a, 1);
  unsigned long long bad = 0, n = 0;
  for (uint32_t xi = blockIdx.x * blockDim.x + threadIdx.x; xi < (1u << 23); xi += gridDim.x * blockDim.x) {
    const float x = __uint_as_float(0x3f800000u | xi);
    const float q = bwd::div_fast(d, x);
    const float e = __fdiv_rn(x, a);
    ++n;
    if (__float_as_uint(q) != __float_as_uint(e)) { ++bad; record(x, a); }
    const float qn = bwd::div_fast(d, -x);
    if (__float_as_uint(qn) != (__float_as_uint(e) ^ 0x80000000u)) { ++bad; record(-x, a); }
    // the packed routine, one lane each sign
    const float2 q2 = bwd::div_fast2(d, make_float2(x, -x));
    if (__float_as_uint(q2.x) != __float_as_uint(e) || __float_as_uint(q2.y) != (__float_as_uint(e) ^ 0x80000000u)) {
      ++bad;
      record(x, a);
    }
  }
  atomicAdd(&g_bad, bad);
  atomicAdd(&g_checked, 2 * n);
}

// The unscaled forms on one (x, a) pair with unscaled_ok(a): exact for
// |x/a| >= 2^-64, bounded below that.  Returns false on a failure.
__device__ bool check_unscaled(float x, float a, float y, float e) {
  const float q = bwd::div_unscaled(x, a, y);
  const float2 q2 = bwd::div_unscaled2(make_float2(x, -x), a, y);
  if (fabsf(e) >= 0x1p-64f)
    return __float_as_uint(q) == __float_as_uint(e) && __float_as_uint(q2.x) == __float_as_uint(e) &&
           __float_as_uint(q2.y) == (__float_as_uint(e) ^ 0x80000000u);
  return fabsf(q) < 0x1p-63f && fabsf(q2.x) < 0x1p-63f && fabsf(q2.y) < 0x1p-63f &&
         fabsf(__fmul_rn(x, y)) < 0x1p-62f;
}

// grid as part1; divisor exponent field ea, dividend exponent field ea + dq
__global__ void part3(uint32_t a_lo, uint32_t ea, int dq) {
  const uint32_t ai = a_lo + blockIdx.y;
  if (ai >= (1u << 23)) return;
  const float a = __uint_as_float((ea << 23) | ai);
  const float y = __frcp_rn(a);
  const uint32_t ex = static_cast<uint32_t>(static_cast<int>(ea) + dq);
  unsigned long long bad = 0, n = 0;
  if (!bwd::unscaled_ok(a)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) { atomicAdd(&g_bad, 1ull); record(0.0f, a); }
    return;
  }
  for (uint32_t xi = blockIdx.x * blockDim.x + threadIdx.x; xi < (1u << 23); xi += gridDim.x * blockDim.x) {
    const float x = __uint_as_float((ex << 23) | xi);
    const float e = __fdiv_rn(x, a);
    n += 2;
    if (!check_unscaled(x, a, y, e)) { ++bad; record(x, a); }
    if (!check_unscaled(-x, a, y, -e)) { ++bad; record(-x, a); }
  }
  atomicAdd(&g_bad, bad);
  atomicAdd(&g_checked, n);
}

__device__ uint32_t hash(uint32_t x) {
  x ^= x >> 16; x *= 0x7feb352dU; x ^= x >> 15; x *= 0x846ca68bU; x ^= x >> 16; return x;
}

__global__ void part2(uint32_t seed, uint32_t iters) {
  unsigned long long bad = 0, n = 0;
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
  for (uint32_t it = 0; it < iters; ++it) {
    const uint32_t h1 = hash(seed ^ hash(tid * 2654435761u + it));
    const uint32_t h2 = hash(h1 + 0x9e3779b9u);
    const uint32_t h3 = hash(h2 + 0x85ebca6bu);
    const uint32_t ea = 1 + (h3 % 253u);                 // divisor exponent field 1..253
    const int dx = -int((h3 >> 8) % 70u);                // quotient exponent 0 .. -69
    int ex = int(ea) + dx;
    if (ex < 1) ex = 1;
    const float a = __uint_as_float((ea << 23) | (h1 & 0x7fffffu));
    const float x = __uint_as_float(((uint32_t)ex << 23) | (h2 & 0x7fffffu) | (h3 & 0x80000000u));
    const float e = __fdiv_rn(x, a);
    const bwd::Divisor d = bwd::make_divisor(a, 1);
    if (bwd::unscaled_ok(a)) {
      ++n;
      if (!check_unscaled(x, a, __frcp_rn(a), e)) { ++bad; record(x, a); }
    }
    if (fabsf(e) < 0x1p-64f) continue;
    if (!d.fast) continue;
    const float q = bwd::div_fast(d, x);
    const float2 q2 = bwd::div_fast2(d, make_float2(x, x));
    ++n;
    if (__float_as_uint(q) != __float_as_uint(e) || __float_as_uint(q2.x) != __float_as_uint(e) ||
        __float_as_uint(q2.y) != __float_as_uint(e)) { ++bad; record(x, a); }
  }
  atomicAdd(&g_bad, bad);
  atomicAdd(&g_checked, n);
}

int main(int argc, char** argv) {
  const uint32_t a_count = argc > 1 ? (uint32_t)atoi(argv[1]) : (1u << 23);
  const uint32_t a_first = argc > 2 ? (uint32_t)atoi(argv[2]) : 0u;
  unsigned long long zero = 0;
  uint32_t z32 = 0;
  cudaMemcpyToSymbol(g_bad, &zero, sizeof zero);
  cudaMemcpyToSymbol(g_checked, &zero, sizeof zero);
  cudaMemcpyToSymbol(g_nfirst, &z32, sizeof z32);
  const uint32_t chunk = 8192;  // divisor significands per launch
  for (uint32_t lo = a_first; lo < a_first + a_count; lo += chunk) {
    dim3 grid(64, chunk < a_first + a_count - lo ? chunk : a_first + a_count - lo);
    part1<<<grid, 256>>>(lo);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { printf("launch error %s\n", cudaGetErrorString(e)); return 2; }
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 2; }
  unsigned long long bad, checked;
  cudaMemcpyFromSymbol(&bad, g_bad, sizeof bad);
  cudaMemcpyFromSymbol(&checked, g_checked, sizeof checked);
  printf("part1: divisor significands %u, checked %llu, mismatches %llu\n", a_count, checked, bad);
  cudaMemcpyToSymbol(g_bad, &zero, sizeof zero);
  cudaMemcpyToSymbol(g_checked, &zero, sizeof zero);
  for (uint32_t s = 0; s < 16; ++s) part2<<<1024, 256>>>(0x1234567u + s * 7919u, 4096);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 2; }
  cudaMemcpyFromSymbol(&bad, g_bad, sizeof bad);
  cudaMemcpyFromSymbol(&checked, g_checked, sizeof checked);
  printf("part2: random exponents, checked %llu, mismatches %llu\n", checked, bad);
  cudaMemcpyToSymbol(g_bad, &zero, sizeof zero);
  cudaMemcpyToSymbol(g_checked, &zero, sizeof zero);
  const uint32_t eas[2] = {89u, 252u};
  const int dqs[3] = {-65, -64, -63};
  for (uint32_t ea : eas)
    for (int dq : dqs)
      for (uint32_t lo = a_first; lo < a_first + a_count; lo += chunk) {
        dim3 grid(64, chunk < a_first + a_count - lo ? chunk : a_first + a_count - lo);
        part3<<<grid, 256>>>(lo, ea, dq);
      }
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 2; }
  cudaMemcpyFromSymbol(&bad, g_bad, sizeof bad);
  cudaMemcpyFromSymbol(&checked, g_checked, sizeof checked);
  printf("part3: unscaled at the range ends, checked %llu, mismatches %llu\n", checked, bad);
  uint32_t nf = 0, first[64];
  cudaMemcpyFromSymbol(&nf, g_nfirst, sizeof nf);
  cudaMemcpyFromSymbol(first, g_first, sizeof first);
  for (uint32_t k = 0; k < nf && k < 32; ++k) {
    float x, a;
    memcpy(&x, &first[2 * k], 4);
    memcpy(&a, &first[2 * k + 1], 4);
    printf("  mismatch x=%a a=%a\n", x, a);
  }
  return (nf == 0) ? 0 : 1;
}
