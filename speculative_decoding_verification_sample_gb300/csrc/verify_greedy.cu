// Greedy verification kernel (spec_verify_greedy).
//
// Method ("devpost.com - phoenix", "What it does"): tokens are kept up to the
// first disagreement between the draft token and the target's argmax, where
// the target's own token is written; the output equals the target decoding
// alone. Ties in the argmax go to the lowest vocabulary index.
//
// GB300 mapping: as the sampling kernel, one cluster per batch row with the
// vocabulary split over its CTAs; each CTA streams its slice of target rows
// 0..K-1 through the bulk-copy ring keeping a running (max, first index) per
// thread; partials are all-gathered over distributed shared memory; a warp
// ballot finds the first mismatch; target row K is streamed only for rows that
// accept all K drafts. Raw logits are compared exactly (no temperature).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "../../include/specverify.h"
#include "cluster_launch.cuh"
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "stream.cuh"

namespace sv {
namespace {

constexpr int kUnroll = 4;

struct Misc {
  int tok[kMaxK];
  int bad_token;
  int abort;
  int first_mismatch;
  int best_idx[kMaxK + 1];
  float src[4];
};

struct Layout {
  Ring ring;
  Xc xc;
  Misc* misc;
  float* wM;      // [R][kCW] best value per warp
  int* wI;        // [R][kCW] its index (-2: NaN seen)
  float* stage;   // exchange payload staging [2R]
};

__host__ __device__ inline int gxc_floats(int R) { return 2 * R > 4 ? 2 * R : 4; }

__host__ __device__ inline size_t greedy_smem_bytes(int R) {
  size_t o = size_t(kStages) * kChunk;
  o += (2 * kStages + 2) * 8;
  o += (sizeof(Misc) + 15) / 16 * 16;
  o += size_t(R) * kCW * 8;
  o += size_t(2) * R * 4;
  o += size_t(2) * kMaxCluster * gxc_floats(R) * 4;
  return (o + 127) / 128 * 128;
}

__device__ inline Layout make_layout(uint8_t* base, int R) {
  Layout L;
  size_t o = size_t(kStages) * kChunk;
  L.ring.buf = base;
  L.ring.full = reinterpret_cast<uint64_t*>(base + o);
  L.ring.empty = L.ring.full + kStages;
  L.xc.bar = L.ring.empty + kStages;
  o += (2 * kStages + 2) * 8;
  L.misc = reinterpret_cast<Misc*>(base + o);
  L.ring.abort = &L.misc->abort;
  o += (sizeof(Misc) + 15) / 16 * 16;
  L.wM = reinterpret_cast<float*>(base + o);
  L.wI = reinterpret_cast<int*>(L.wM + R * kCW);
  o += size_t(R) * kCW * 8;
  L.stage = reinterpret_cast<float*>(base + o);
  o += size_t(2) * R * 4;
  L.xc.buf = reinterpret_cast<float*>(base + o);
  L.xc.slot = gxc_floats(R);
  return L;
}

// (value, index) order: larger value first, then smaller index.
__device__ __forceinline__ bool better(float b, int i, float best, int idx) {
  return b > best || (b == best && i < idx);
}

template <class E>
struct ArgmaxOp {
  float best;
  int idx;
  int bad;
  int row_base;
  const Layout* L;
  __device__ void begin_row(int) {
    best = -INFINITY;
    idx = INT_MAX;
    bad = 0;
  }
  // Vectors arrive in increasing index order per thread, so a strict '>' keeps
  // the first occurrence of the maximum.
  __device__ __forceinline__ void vec(const uint4& v, int vi) {
    const float vm = E::vmax(v);
    if (vm != vm) {
      bad = 1;
      return;
    }
    if (vm > best || idx == INT_MAX) {
      float z[E::kVec];
      E::unpack(v, z);
      int k = 0;
#pragma unroll
      for (int kk = E::kVec - 1; kk >= 0; --kk)
        if (z[kk] == vm) k = kk;
      best = vm;
      idx = vi * E::kVec + k;
    }
  }
  __device__ void end_row(int r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (better(ob, oi, best, idx)) {
        best = ob;
        idx = oi;
      }
    }
    const int anybad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      const int rr = row_base + r;
      L->wM[rr * kCW + warp] = best;
      L->wI[rr * kCW + warp] = anybad ? -2 : idx;
    }
  }
};

// Consumers: CTA-level (value, index) of rows [r0, r1) into the payload, then
// the all-gather and the final (value, lowest index) per row in every CTA.
__device__ bool argmax_exchange(const Layout& L, uint32_t& e, int r0, int r1, int crank,
                                int csize) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = r0 + warp; r < r1; r += kCW) {
    float best = lane < kCW ? L.wM[r * kCW + lane] : -INFINITY;
    int idx = lane < kCW ? L.wI[r * kCW + lane] : INT_MAX;
    int bad = (idx == -2);
    if (bad) idx = INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (better(ob, oi, best, idx)) {
        best = ob;
        idx = oi;
      }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      L.stage[2 * (r - r0)] = best;
      L.stage[2 * (r - r0) + 1] = __int_as_float(bad ? -2 : idx);
    }
  }
  consumers_sync();
  if (threadIdx.x < 32) xc_push(L.xc, e, L.stage, 2 * (r1 - r0), crank, csize);
  const bool ok = xc_wait(L.xc, e, L.ring.abort);
  for (int r = r0 + int(threadIdx.x); r < r1 && ok; r += kCons) {
    float best = -INFINITY;
    int idx = INT_MAX, bad = 0;
    for (int q = 0; q < csize; ++q) {
      const float* s = xc_slot(L.xc, e, q) + 2 * (r - r0);
      const int i = __float_as_int(s[1]);
      if (i == -2) {
        bad = 1;
        continue;
      }
      if (better(s[0], i, best, idx)) {
        best = s[0];
        idx = i;
      }
    }
    L.misc->best_idx[r] = (bad || idx == INT_MAX) ? -1 : idx;
  }
  ++e;
  consumers_sync();
  return ok;
}

struct GreedyArgs {
  const void* target;
  const int32_t* tokens;
  int B, K, V;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
};

template <class E>
__device__ void greedy_row(const GreedyArgs& a, const Layout& L, int b, int vbeg, int vend,
                           int crank, int csize, uint32_t& it, uint32_t& e) {
  using T = typename E::T;
  Misc& ms = *L.misc;
  const int K = a.K, V = a.V;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const T* tgt = static_cast<const T*>(a.target) + size_t(b) * (K + 1) * V;
  if (warp == 1) {
    int bad = 0;
    if (lane < K) {
      const int d = a.tokens[size_t(b) * K + lane];
      ms.tok[lane] = d;
      bad = (d < 0 || d >= V);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) ms.bad_token = bad;
  }
  ArgmaxOp<E> op;
  op.row_base = 0;
  op.L = &L;
  it = consume_rows(L.ring, it, K, vbeg, vend, op);
  consumers_sync();
  bool alive = argmax_exchange(L, e, 0, K, crank, csize);
  // first mismatch by warp ballot
  if (warp == 0) {
    const int g = lane < K ? ms.best_idx[lane] : 0;
    const unsigned mism = __ballot_sync(0xffffffffu, lane < K && g != ms.tok[lane]);
    if (lane == 0) ms.first_mismatch = mism ? (__ffs(int(mism)) - 1) : K;
  }
  consumers_sync();
  const int n = ms.first_mismatch;
  bool error = ms.bad_token != 0 || !alive;
  for (int i = 0; i <= min(n, K - 1); ++i)
    if (ms.best_idx[i] < 0) error = true;  // a NaN row up to the first mismatch
  int token = -1;
  if (!error) {
    if (n < K) {
      token = ms.best_idx[n];
    } else {
      // target row K, only for rows that accept all K drafts: direct loads
      const uint4* p = reinterpret_cast<const uint4*>(tgt + size_t(K) * V);
      op.row_base = K;
      op.begin_row(0);
      for (int v0 = vbeg + tid; v0 < vend; v0 += kCons * kUnroll) {
        uint4 buf[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (v0 + u * kCons < vend) buf[u] = ldg_nc_v4(p + v0 + u * kCons);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (v0 + u * kCons < vend) op.vec(buf[u], v0 + u * kCons);
      }
      op.end_row(0);
      consumers_sync();
      alive = argmax_exchange(L, e, K, K + 1, crank, csize);
      token = ms.best_idx[K];
      if (token < 0 || !alive) error = true;
    }
  }
  if (crank == 0) {
    if (tid <= K) {
      int32_t v;
      if (error) v = -1;
      else if (tid < n) v = ms.tok[tid];
      else if (tid == n) v = token;
      else v = -1;
      a.out_tokens[size_t(b) * (K + 1) + tid] = v;
    }
    if (tid == 0) {
      a.out_n[b] = error ? -1 : n;
      if (error && a.err) {
        const int bit = *L.ring.abort ? SPEC_DERR_TIMEOUT
                        : ms.bad_token ? SPEC_DERR_TOKEN
                                       : SPEC_DERR_LOGITS;
        atomicOr(a.err, bit);
      }
    }
  }
  consumers_sync();
}

template <class E>
__global__ void __launch_bounds__(kThreads, 2) verify_greedy_kernel(const GreedyArgs a, int ncl) {
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K, V = a.V, R = K + 1;
  const Layout L = make_layout(smem_raw, R);
  const int crank = int(cluster_ctarank()), csize = int(cluster_nctarank());
  const int cid = blockIdx.x / csize;
  int vbeg, vend;
  cta_slice(V / E::kVec, crank, csize, vbeg, vend);
  ring_xc_init(L.ring, L.xc, csize);
  __syncthreads();
  cluster_sync();
  if (threadIdx.x >= kCons) {
    if (threadIdx.x == kCons) {
      uint32_t it = 0;
      for (int b = cid; b < a.B; b += ncl) {
        const T* tgt = static_cast<const T*>(a.target) + size_t(b) * (K + 1) * V;
        auto rp = [&](int r) -> const T* { return tgt + size_t(r) * V; };
        it = produce_rows(L.ring, it, K, rp, vbeg, vend);
      }
    }
  } else {
    uint32_t it = 0, e = 0;
    for (int b = cid; b < a.B; b += ncl) greedy_row<E>(a, L, b, vbeg, vend, crank, csize, it, e);
  }
  __syncthreads();
  cluster_sync();
}

}  // namespace

int launch_verify_greedy(const GreedyLaunch& g) {
  GreedyArgs a;
  a.target = g.target;
  a.tokens = g.tokens;
  a.B = g.B;
  a.K = g.K;
  a.V = g.V;
  a.out_tokens = g.out_tokens;
  a.out_n = g.out_n;
  a.err = g.err;
  const int kvec = (g.dtype == SPEC_BF16) ? 8 : 4;
  const int csize = pick_cluster(g.B, g.V / kvec);
  const size_t smem = greedy_smem_bytes(g.K + 1);
  cudaStream_t st = static_cast<cudaStream_t>(g.stream);
  if (g.dtype == SPEC_BF16)
    return launch_persistent(verify_greedy_kernel<EBf16>, a, g.B, csize, smem, st);
  return launch_persistent(verify_greedy_kernel<EF32>, a, g.B, csize, smem, st);
}

int verify_cluster_size(int B, int V, int dtype) {
  const int kvec = (dtype == SPEC_BF16) ? 8 : 4;
  return pick_cluster(B, V / kvec);
}

}  // namespace sv
