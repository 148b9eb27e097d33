// Host helper for the persistent launches of the verification kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "../../include/specverify.h"
#include "common.cuh"

namespace sv {

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
  kern<<<grid, kThreads, smem, st>>>(args);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // namespace sv
