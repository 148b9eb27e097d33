// Shared device-side definitions: launch geometry, element traits for bf16 and
// fp32 logits, warp reductions.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace sv {

constexpr int kCW = 8;                 // consumer warps per CTA
constexpr int kCons = kCW * 32;        // consumer threads
constexpr int kThreads = kCons + 64;   // + producer warp (bulk-copy issue) + finisher warp
constexpr int kStages = 3;             // ring depth (3 x 32 KB: two CTAs per SM)
constexpr int kChunk = 32768;          // bytes per ring stage
constexpr int kMaxK = 31;              // draft positions (fits a warp ballot)

constexpr float kU = 5.9604644775390625e-8f;  // fp32 unit roundoff 2^-24
// Largest row offset |ceil(max z * log2(e)/T)| (exclusive) that the sampling
// and top-p paths accept: within it the double-float terms keep their error
// bound; a row beyond it is reported as invalid logits.
constexpr float kMaxOffset = 262144.0f;  // 2^18
constexpr float kLn2f = 0.693147180559945309417232121458176568f;

// max that returns NaN when either input is NaN (PTX max.NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ----------------------------------------------------------------- elements
// bf16 logits: a 16-byte vector holds 8 values; widening to fp32 is exact.
struct EBf16 {
  using T = uint16_t;
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void unpack(const uint4& v, float (&z)[8]) {
    z[0] = __uint_as_float(v.x << 16);
    z[1] = __uint_as_float(v.x & 0xffff0000u);
    z[2] = __uint_as_float(v.y << 16);
    z[3] = __uint_as_float(v.y & 0xffff0000u);
    z[4] = __uint_as_float(v.z << 16);
    z[5] = __uint_as_float(v.z & 0xffff0000u);
    z[6] = __uint_as_float(v.w << 16);
    z[7] = __uint_as_float(v.w & 0xffff0000u);
  }
  // Maximum of the 8 values; NaN if any value is NaN.
  __device__ static __forceinline__ float vmax(const uint4& v) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return max_nan(__low2float(m), __high2float(m));
  }
  __device__ static __forceinline__ float cvt(T x) {
    return __uint_as_float(static_cast<uint32_t>(x) << 16);
  }
  __device__ static __forceinline__ float load(const T* p, int64_t i) { return cvt(p[i]); }
};

// fp32 logits: 4 values per 16-byte vector.
struct EF32 {
  using T = float;
  static constexpr int kVec = 4;
  __device__ static __forceinline__ void unpack(const uint4& v, float (&z)[4]) {
    z[0] = __uint_as_float(v.x);
    z[1] = __uint_as_float(v.y);
    z[2] = __uint_as_float(v.z);
    z[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ float vmax(const uint4& v) {
    float a = __uint_as_float(v.x), b = __uint_as_float(v.y), c = __uint_as_float(v.z),
          d = __uint_as_float(v.w);
    return max_nan(max_nan(a, b), max_nan(c, d));
  }
  __device__ static __forceinline__ float cvt(T x) { return x; }
  __device__ static __forceinline__ float load(const T* p, int64_t i) { return p[i]; }
};

// ----------------------------------------------------------------- warp ops
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Warp sums of N values per lane at once (N a power of two <= 32), by
// recursive halving: at each of the first log2(N) butterfly steps a lane
// keeps half of its values and trades the other half with its partner, so
// the warp issues N - 1 + 5 - log2(N) shuffles instead of 5 N. The sum of
// slot k ends on the lanes l with l >> (5 - log2 N) == k; the additions pair
// the same lanes as warp_sum_f, so each slot's sum equals warp_sum_f of it.
template <int N>
__device__ __forceinline__ float warp_sum_slots(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; (N >> (t + 1)) >= 1; ++t) {
    const int h = N >> (t + 1), o = 16 >> t;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int o = 16 / N; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  return v[0];
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 2^k for an integer-valued float k in [-126, 127]; 0 below.
__device__ __forceinline__ float pow2i(float k) {
  int ki = static_cast<int>(k);
  if (ki < -126) return 0.0f;
  return __int_as_float((ki + 127) << 23);
}

// Integer softmax offset for a maximum m: ceil(m * c). Any integer works as the
// offset of exp2(z*c - offset); taking it from the row maximum keeps every
// term <= 2 and the largest >= 1/2. Computed the same way everywhere so that
// equal maxima give bit-identical offsets.
__device__ __forceinline__ float offset_of(float m, float c) { return ceilf(__fmul_rn(m, c)); }

}  // namespace sv
