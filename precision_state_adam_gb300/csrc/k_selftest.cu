// Self-test of the update's correctly rounded root and quotient (sqrt2_rn, div2_rn and the
// domain switch in adamw_n) against the hardware's IEEE sqrt and division.
#include "psadam_kernels.cuh"

namespace psadam {

// mismatch counters: [0] root, [1] quotient significands, [2] exponent scaling of the
// approximations, [3] the whole update through adamw_n against the per-element IEEE update
static __device__ unsigned long long g_math_mismatch[4];

__global__ void psadam_math_zero_kernel() {
  if (threadIdx.x < 4) g_math_mismatch[threadIdx.x] = 0ULL;
}

// Every float in [2^-102, 2^128): exponent fields 25..254, all significands, two per thread
// and call (one in each lane of the pair).
__global__ void psadam_math_root_kernel() {
  constexpr unsigned long long kPairs = (230ULL << 23) / 2;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  unsigned long long bad = 0;
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < kPairs; i += stride) {
    const uint32_t b0 = (25u << 23) + (uint32_t)(2 * i);
    const float v0 = __uint_as_float(b0), v1 = __uint_as_float(b0 + 1u);
    const float2 s = sqrt2_rn(make_float2(v0, v1));
    bad += (__float_as_uint(s.x) != __float_as_uint(__fsqrt_rn(v0))) +
           (__float_as_uint(s.y) != __float_as_uint(__fsqrt_rn(v1)));
  }
  if (bad) atomicAdd(&g_math_mismatch[0], bad);
}

// a, b in [1, 2): every significand of b (one per thread), significands a0 + k*step of a
// (k < 2*na, in pairs).
__global__ void psadam_math_quot_kernel(uint32_t a0, uint32_t step, uint32_t na) {
  const uint32_t mb = blockIdx.x * blockDim.x + threadIdx.x;
  if (mb >= (1u << 23)) return;
  const float b = __uint_as_float(0x3F800000u | mb);
  unsigned long long bad = 0;
  for (uint32_t k = 0; k < na; ++k) {
    const float x0 = __uint_as_float(0x3F800000u | ((a0 + (2 * k) * step) & 0x7FFFFFu));
    const float x1 = __uint_as_float(0x3F800000u | ((a0 + (2 * k + 1) * step) & 0x7FFFFFu));
    const float2 q = div2_rn(make_float2(x0, x1), f2(b));
    bad += (__float_as_uint(q.x) != __float_as_uint(__fdiv_rn(x0, b))) +
           (__float_as_uint(q.y) != __float_as_uint(__fdiv_rn(x1, b)));
  }
  if (bad) atomicAdd(&g_math_mismatch[1], bad);
}

// rcp~(b * 2^k) = rcp~(b) * 2^-k for k in [-120, 120] and rsqrt~(v * 4^h) = rsqrt~(v) * 2^-h
// for v in [1, 4), h in [-60, 60]: every significand.
__global__ void psadam_math_scale_kernel() {
  const uint32_t mb = blockIdx.x * blockDim.x + threadIdx.x;
  if (mb >= (1u << 23)) return;
  const float b = __uint_as_float(0x3F800000u | mb), b2 = __fmul_rn(b, 2.0f);
  const float r = rcp_approx(b), s = rsqrt_approx(b), s2 = rsqrt_approx(b2);
  unsigned long long bad = 0;
  for (int k = -120; k <= 120; ++k) bad += __float_as_uint(rcp_approx(ldexpf(b, k))) != __float_as_uint(ldexpf(r, -k));
  for (int h = -60; h <= 60; ++h) {
    bad += __float_as_uint(rsqrt_approx(ldexpf(b, 2 * h))) != __float_as_uint(ldexpf(s, -h));
    bad += __float_as_uint(rsqrt_approx(ldexpf(b2, 2 * h))) != __float_as_uint(ldexpf(s2, -h));
  }
  if (bad) atomicAdd(&g_math_mismatch[2], bad);
}

// SplitMix64's output function (Steele, Lea and Flood, OOPSLA 2014): a counter to 64 bits.
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
// A float of random sign and significand with exponent e0 + (r % span).
__device__ __forceinline__ float rand_float(uint64_t r, int e0, int span) {
  const uint32_t e = (uint32_t)(127 + e0 + (int)((r >> 40) % (uint64_t)span));
  return __uint_as_float(((uint32_t)(r >> 63) << 31) | (e << 23) | (uint32_t)(r & 0x7FFFFFu));
}

// The update of 8 elements per thread through adamw_n (the fused root and quotient where
// the thread's elements allow them) against adamw_element (IEEE per element), bit for bit.
// Seven tiles in eight draw grads and moments inside the fused domain; the eighth draws them
// over far wider exponent ranges, with zeros, so that the domain switch goes both ways.
__global__ void psadam_math_update_kernel(StepConsts c, unsigned long long seed, unsigned long long tiles) {
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  unsigned long long bad = 0;
  for (unsigned long long t = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; t < tiles; t += stride) {
    float p[8], g[8], m[8], v[8], p1[8], m1[8], v1[8];
    const bool wide = (mix64(seed ^ (t * 0x100000001B3ULL)) & 7) == 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const unsigned long long e = 4 * (8 * t + i);
      const uint64_t r0 = mix64(seed + e), r1 = mix64(seed + e + 1), r2 = mix64(seed + e + 2), r3 = mix64(seed + e + 3);
      p[i] = rand_float(r0, -12, 12);
      if (wide) {
        g[i] = (r3 & 7) == 0 ? 0.0f : rand_float(r1, -80, 120);
        m[i] = (r3 & 0x70) == 0 ? 0.0f : rand_float(r2, -120, 180);
        v[i] = (r3 & 0x700) == 0 ? 0.0f : fabsf(rand_float(r3 >> 12, -126, 166));
      } else {
        g[i] = rand_float(r1, -30, 30);
        m[i] = rand_float(r2, -45, 40);
        v[i] = fabsf(rand_float(r3, -50, 40));
      }
      p1[i] = p[i];
      m1[i] = m[i];
      v1[i] = v[i];
    }
    adamw_n<true, 8>(p, g, m, v, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      adamw_element<true>(p1[i], g[i], m1[i], v1[i], c);
      bad += (__float_as_uint(p[i]) != __float_as_uint(p1[i])) + (__float_as_uint(m[i]) != __float_as_uint(m1[i])) +
             (__float_as_uint(v[i]) != __float_as_uint(v1[i]));
    }
  }
  if (bad) atomicAdd(&g_math_mismatch[3], bad);
}

cudaError_t launch_math_selftest(int full, const StepConsts* c, int n_c, unsigned long long* out, cudaStream_t s) {
  constexpr int kT = 256;
  constexpr int kGrid = 152 * 8;
  psadam_math_zero_kernel<<<1, 32, 0, s>>>();
  psadam_math_root_kernel<<<kGrid, kT, 0, s>>>();
  psadam_math_scale_kernel<<<(1 << 23) / kT, kT, 0, s>>>();
  // every significand of a (2^23, in 2^14 launches of 512) or 8192 of them spread over the range
  const uint32_t n_a = full ? (1u << 23) : 8192u, step = full ? 1u : (1u << 23) / 8192u;
  constexpr uint32_t kPerLaunch = 512;
  for (uint32_t k0 = 0; k0 < n_a; k0 += kPerLaunch) {
    psadam_math_quot_kernel<<<(1 << 23) / kT, kT, 0, s>>>(k0 * step + (full ? 0u : 4099u), step, kPerLaunch / 2);
    if (full && (k0 / kPerLaunch) % 64 == 63) {  // keep the queue short on the long run
      const cudaError_t e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return e;
    }
  }
  for (int i = 0; i < n_c; ++i) psadam_math_update_kernel<<<kGrid, kT, 0, s>>>(c[i], 0x5EEDULL + i, 1ULL << 22);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(out, g_math_mismatch, sizeof(g_math_mismatch), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}
}  // namespace psadam
