// Host helper for the persistent launches of the verification kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "../../include/specverify.h"
#include "common.cuh"

namespace sv {

// Launch with programmatic stream serialization (see pdl_wait): the kernel
// may start while its predecessor on the stream finishes, and waits for it
// with pdl_wait() before touching that predecessor's results.
template <class Kern, class... Args>
int launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return SPEC_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// Zeroes n 16-byte words of the workspace (the per-launch counters and work
// queue) ahead of a verification launch, which starts early and waits for it
// (programmatic dependent launch) instead of following a host memset.
static __global__ void zero_words_kernel(uint4* p, size_t n) {
  pdl_trigger();
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += size_t(gridDim.x) * blockDim.x)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

inline int zero_workspace(void* ws, size_t bytes, cudaStream_t st) {
  const size_t n = (bytes + 15) / 16;  // the zeroed regions are 256-byte aligned and padded
  const int grid = int((n + 255) / 256 < 512 ? (n + 255) / 256 : 512);
  zero_words_kernel<<<grid > 0 ? grid : 1, 256, 0, st>>>(static_cast<uint4*>(ws), n);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// Dataflow launch: one grid of persistent CTAs, as many as are co-resident
// (occupancy query, cached per kernel and shared-memory size); the kernels
// fetch their work from the workspace counters.
template <class Kern, class Args>
int launch_dataflow(Kern kern, const Args& args, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return SPEC_ECUDA;
  // Occupancy per (kernel, shared memory, device), cached for the process;
  // the mutex lets several host threads launch at once.
  struct Entry {
    const void* k;
    size_t s;
    int dev, grid;
  };
  static Entry cache[16];
  static int ncache = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ECUDA;
  int grid = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ncache; ++i)
      if (cache[i].k == reinterpret_cast<const void*>(kern) && cache[i].s == smem &&
          cache[i].dev == dev)
        grid = cache[i].grid;
  }
  if (grid == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess || per_sm < 1) return SPEC_ENOTSUP;
    grid = sms * per_sm;
    std::lock_guard<std::mutex> lock(mu);
    if (ncache < 16) cache[ncache++] = {reinterpret_cast<const void*>(kern), smem, dev, grid};
  }
  if (const char* env = std::getenv("SPECVERIFY_GRID")) {
    const int g = std::atoi(env);
    if (g > 0 && g < grid) grid = g;
  }
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, args);
}

}  // namespace sv
