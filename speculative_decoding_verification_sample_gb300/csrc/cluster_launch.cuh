// Host helpers for the cluster launches of the verification kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstdlib>

#include "../../include/specverify.h"
#include "common.cuh"

namespace sv {

// CTAs per batch row: 16 (the vocabulary split 16 ways keeps a CTA's slice of
// a 152k-token row at 19 KB of bf16). Environment override SPECVERIFY_CLUSTER in
// {1,2,4,8,16}; never more CTAs than 16-byte vectors in a row.
inline int pick_cluster(int B, int nvec) {
  (void)B;
  int c = 16;
  if (const char* e = std::getenv("SPECVERIFY_CLUSTER")) c = std::atoi(e);
  if (c != 1 && c != 2 && c != 4 && c != 8 && c != 16) c = 16;
  while (c > 1 && c > nvec) c >>= 1;
  return c;
}

// Launches `kern` on B clusters of `csize` CTAs (kThreads threads each).
template <class Kern, class Args>
int launch_cluster(Kern kern, const Args& args, int B, int csize, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return SPEC_ECUDA;
  if (csize > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return SPEC_ECUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B) * unsigned(csize), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(csize);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, args);
  return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// Persistent launch: as many clusters of `csize` CTAs as can be co-resident
// (queried once per kernel and configuration), at most B; the kernel receives
// the cluster count and strides over the batch rows.
template <class Kern, class Args>
int launch_persistent(Kern kern, const Args& args, int B, int csize, size_t smem,
                      cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return SPEC_ECUDA;
  if (csize > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return SPEC_ECUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(csize);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // cache of co-resident cluster counts, keyed by kernel, cluster size and smem
  struct Entry {
    const void* k;
    int c;
    size_t s;
    int n;
  };
  static Entry cache[16];
  static int ncache = 0;
  int ncl = 0;
  for (int i = 0; i < ncache; ++i)
    if (cache[i].k == reinterpret_cast<const void*>(kern) && cache[i].c == csize && cache[i].s == smem)
      ncl = cache[i].n;
  if (ncl == 0) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3(unsigned(sms / csize * csize > 0 ? sms / csize * csize : csize), 1, 1);
    e = cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg);
    if (e != cudaSuccess || ncl < 1) return SPEC_ENOTSUP;
    if (ncache < 16) cache[ncache++] = {reinterpret_cast<const void*>(kern), csize, smem, ncl};
  }
  if (const char* env = std::getenv("SPECVERIFY_MAX_CLUSTERS")) {
    const int m = std::atoi(env);
    if (m > 0 && m < ncl) ncl = m;
  }
  if (ncl > B) ncl = B;
  cfg.gridDim = dim3(unsigned(ncl) * unsigned(csize), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, args, ncl);
  return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // namespace sv
