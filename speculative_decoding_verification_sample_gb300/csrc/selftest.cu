// Self-test: maximum relative error of the hardware base-2 exponential
// (ex2.approx.ftz.f32) over every fp32 argument in [lo, hi], against the
// fp64 exp2 of the same argument. The certified fp32 path of the sampler uses
// a bound above this maximum (launch.h, kEx2RelErrBound); this entry point lets
// the tests re-measure it on the GPU the library runs on.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/specverify.h"
#include "ptx.cuh"

namespace sv {

__global__ void ex2_error_kernel(uint32_t lo_bits, uint64_t count, int negative,
                                 unsigned long long* out_max_bits) {
  double worst = 0.0;
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride) {
    const uint32_t bits = lo_bits + uint32_t(i);
    const float x = __uint_as_float(negative ? (bits | 0x80000000u) : bits);
    const double ref = exp2(double(x));
    const double got = double(ex2_approx(x));
    const double rel = fabs(got - ref) / ref;
    worst = fmax(worst, rel);
  }
  for (int o = 16; o > 0; o >>= 1) worst = fmax(worst, __shfl_xor_sync(0xffffffffu, worst, o));
  if ((threadIdx.x & 31) == 0)
    atomicMax(out_max_bits, static_cast<unsigned long long>(__double_as_longlong(worst)));
}

}  // namespace sv

extern "C" int spec_selftest_ex2(float lo, float hi, double* out_max_rel, void* stream) {
  if (!out_max_rel || !(lo <= hi) || lo < -126.0f || hi > 127.0f) return SPEC_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* out = reinterpret_cast<unsigned long long*>(out_max_rel);
  if (cudaMemsetAsync(out, 0, sizeof(double), st) != cudaSuccess) return SPEC_ECUDA;
  // negative part [lo, min(hi, -0)] and non-negative part [max(lo, 0), hi], as magnitude bit ranges
  auto run = [&](float a, float b, int neg) -> int {
    uint32_t ua, ub;
    memcpy(&ua, &a, 4);
    memcpy(&ub, &b, 4);
    ua &= 0x7fffffffu;
    ub &= 0x7fffffffu;
    if (ua > ub) {
      const uint32_t t = ua;
      ua = ub;
      ub = t;
    }
    sv::ex2_error_kernel<<<1216, 256, 0, st>>>(ua, uint64_t(ub) - ua + 1, neg, out);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
  };
  int s = SPEC_OK;
  if (lo < 0.0f) s = run(lo, hi < 0.0f ? hi : -0.0f, 1);
  if (s == SPEC_OK && hi >= 0.0f) s = run(lo > 0.0f ? lo : 0.0f, hi, 0);
  return s;
}
