// Row-slice streaming and cluster exchanges shared by the verification kernels.
//
// Streaming. A CTA owns a contiguous slice of 16-byte vectors of every logit
// row it visits. One producer thread (lane 0 of the last warp) issues 1-D bulk
// async copies global -> shared into a kStages-deep ring of kChunk-byte
// stages, each completing on its "full" mbarrier; the kCW consumer warps read a
// stage, then arrive on its "empty" mbarrier so the producer may refill it.
// The kernels are persistent: the producer walks the same sequence of rows as
// the consumers and runs ahead of them by up to the ring's capacity, so the
// next batch row is already in flight while the consumers finish the current
// one.
//
// Exchanges. Values that every CTA of the cluster needs (per-CTA partial sums,
// the drawn token) are all-gathered through distributed shared memory: each
// CTA stores its slot into every CTA and arrives remotely on that CTA's
// exchange mbarrier; every CTA waits for C arrivals. Two buffers alternate, so
// slot e+2 can only be rewritten after every CTA has passed exchange e+1 and
// therefore finished reading exchange e. The producer never joins these
// synchronisations, which is what lets it keep streaming.
//
// All waits are bounded; a timeout sets an abort flag, later waits return at
// once and the kernel reports SPEC_DERR_TIMEOUT instead of hanging.
#pragma once
#include <cstdint>

#include "../../include/specverify.h"
#include "common.cuh"
#include "ptx.cuh"

namespace sv {

struct Ring {
  uint8_t* buf;         // kStages * kChunk bytes
  uint64_t* full;       // [kStages]
  uint64_t* empty;      // [kStages]
  volatile int* abort;  // shared flag
};

struct Xc {
  float* buf;     // [2][kMaxCluster][slot]
  uint64_t* bar;  // [2], expected arrivals: cluster size
  int slot;       // floats per CTA slot
};

// Barrier among the consumer warps only.
__device__ __forceinline__ void consumers_sync() { named_bar_sync(1, kCons); }

__device__ inline void ring_xc_init(const Ring& r, const Xc& x, int csize) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], kCW);
    }
    mbar_init(&x.bar[0], csize);
    mbar_init(&x.bar[1], csize);
    *r.abort = 0;
    fence_mbar_init();
  }
}

// Chunking of a row slice of nv vectors: nchunk chunks of cv vectors (cv*16 <= kChunk).
__device__ __forceinline__ void chunking(int nv, int& nchunk, int& cv) {
  nchunk = nv > 0 ? (nv * 16 + kChunk - 1) / kChunk : 0;
  cv = nchunk > 0 ? (nv + nchunk - 1) / nchunk : 0;
}

// Producer side: issue the copies of `nrows` row slices. Returns the new counter.
template <class RowPtr>
__device__ uint32_t produce_rows(const Ring& ring, uint32_t it, int nrows, RowPtr rowptr,
                                 int vbeg, int vend) {
  int nchunk, cv;
  chunking(vend - vbeg, nchunk, cv);
  for (int r = 0; r < nrows; ++r) {
    const char* row = reinterpret_cast<const char*>(rowptr(r));
    for (int k = 0; k < nchunk; ++k, ++it) {
      const int stage = it % kStages;
      if (it >= kStages) {
        if (*ring.abort || !mbar_wait(&ring.empty[stage], ((it / kStages) - 1) & 1)) {
          *ring.abort = 1;
          return it;
        }
      }
      const int c0 = vbeg + k * cv;
      const int c1 = min(vend, c0 + cv);
      const uint32_t bytes = uint32_t(c1 - c0) * 16u;
      mbar_arrive_expect_tx(&ring.full[stage], bytes);
      bulk_g2s(ring.buf + size_t(stage) * kChunk, row + size_t(c0) * 16, bytes, &ring.full[stage]);
    }
  }
  return it;
}

// Consumer side: op.begin_row(r), op.vec(vector, vector_index) for every vector,
// op.end_row(r) (warp-collective) for each of `nrows` row slices.
template <class Op>
__device__ uint32_t consume_rows(const Ring& ring, uint32_t it, int nrows, int vbeg, int vend,
                                 Op& op) {
  const int tid = threadIdx.x, lane = tid & 31;
  int nchunk, cv;
  chunking(vend - vbeg, nchunk, cv);
  for (int r = 0; r < nrows; ++r) {
    op.begin_row(r);
    for (int k = 0; k < nchunk; ++k, ++it) {
      const int stage = it % kStages;
      if (*ring.abort || !mbar_wait(&ring.full[stage], (it / kStages) & 1)) {
        *ring.abort = 1;
        continue;
      }
      const int c0 = vbeg + k * cv;
      const int c1 = min(vend, c0 + cv);
      const uint4* buf = reinterpret_cast<const uint4*>(ring.buf + size_t(stage) * kChunk);
      for (int i = tid; i < c1 - c0; i += kCons) op.vec(buf[i], c0 + i);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ring.empty[stage]);
    }
    op.end_row(r);
  }
  return it;
}

// ---------------------------------------------------------------- exchanges
__device__ __forceinline__ float* xc_slot(const Xc& x, uint32_t e, int q) {
  return x.buf + (size_t(e & 1) * kMaxCluster + q) * x.slot;
}

// Warp 0 of the consumers: push this CTA's n floats (local `src`) into slot
// [crank] of every CTA and arrive on their exchange barriers.
__device__ __forceinline__ void xc_push(const Xc& x, uint32_t e, const float* src, int n,
                                        int crank, int csize) {
  const int lane = threadIdx.x & 31;
  if (lane < csize) {
    const uint32_t q = lane;
    const uint32_t dst = smem_u32(xc_slot(x, e, crank));
    for (int i = 0; i < n; ++i) st_cluster_f32(mapa_shared(dst + 4u * i, q), src[i]);
    mbar_arrive_remote(mapa_shared(smem_u32(&x.bar[e & 1]), q));
  }
}

// Consumers: wait until every CTA's slot of exchange e has arrived.
__device__ __forceinline__ bool xc_wait(const Xc& x, uint32_t e, volatile int* abort) {
  if (*abort) return false;
  if (!mbar_wait_cluster(&x.bar[e & 1], (e >> 1) & 1)) {
    *abort = 1;
    return false;
  }
  return true;
}

// The CTA's slice of a row of `nvec` vectors when C CTAs split it.
__device__ __forceinline__ void cta_slice(int nvec, int crank, int csize, int& vbeg, int& vend) {
  vbeg = int(int64_t(nvec) * crank / csize);
  vend = int(int64_t(nvec) * (crank + 1) / csize);
}

}  // namespace sv
