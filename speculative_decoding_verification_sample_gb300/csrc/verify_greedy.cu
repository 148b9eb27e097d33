// Greedy verification kernel (spec_verify_greedy).
//
// Method ("devpost.com - phoenix", "What it does"): tokens are kept up to the
// first disagreement between the draft token and the target's argmax, where
// the target's own token is written; the output equals the target decoding
// alone. Ties in the argmax go to the lowest vocabulary index.
//
// GB300 mapping (dataflow engine, engine.cuh): task (b, s) streams slice s of
// target rows 0..K-1 and leaves each row's (max, first index) in the
// workspace; the CTA completing row b combines the S partials, finds the first
// mismatch with a warp ballot, and either writes the row or (all K accepted)
// enqueues the slices of target row K, whose completing CTA writes the bonus
// token. Raw logits are compared exactly (no temperature).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "../../include/specverify.h"
#include "common.cuh"
#include "engine.cuh"
#include "launch_util.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace sv {
namespace {

enum { kG1 = 1, kGB = 2 };

struct GreedyArgs {
  const void* target;
  const int32_t* tokens;
  int B, K, V, S, nvec;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  Ws ws;
};

struct Misc {
  int abort;
  int last;
  int tok[kMaxK];
  int best[kMaxK + 1];
  int first_mismatch;
  int bad_token;
};

struct Smem {
  Ring ring;
  Misc* misc;
  float* wM;  // [K+1][kCW]
  int* wI;    // [K+1][kCW]  (-2: NaN seen)
};

__host__ __device__ inline size_t greedy_smem_bytes(int R) {
  size_t o = size_t(kStages) * kChunk;
  o += 2 * kStages * 8;
  o += kStages * sizeof(ChunkMeta) + kStages * sizeof(QTask);
  o += (sizeof(Misc) + 15) / 16 * 16;
  o += size_t(R) * kCW * 8;
  return (o + 127) / 128 * 128;
}

__device__ inline Smem make_smem(uint8_t* base, int R) {
  Smem L;
  size_t o = size_t(kStages) * kChunk;
  L.ring.buf = base;
  L.ring.full = reinterpret_cast<uint64_t*>(base + o);
  L.ring.empty = L.ring.full + kStages;
  o += 2 * kStages * 8;
  L.ring.meta = reinterpret_cast<ChunkMeta*>(base + o);
  o += kStages * sizeof(ChunkMeta);
  L.ring.ttab = reinterpret_cast<QTask*>(base + o);
  o += kStages * sizeof(QTask);
  L.misc = reinterpret_cast<Misc*>(base + o);
  L.ring.abort = &L.misc->abort;
  o += (sizeof(Misc) + 15) / 16 * 16;
  L.wM = reinterpret_cast<float*>(base + o);
  L.wI = reinterpret_cast<int*>(L.wM + R * kCW);
  return L;
}

// (value, index) order: larger value first, then smaller index.
__device__ __forceinline__ bool better(float b, int i, float best, int idx) {
  return b > best || (b == best && i < idx);
}

template <class E>
struct ArgmaxOp {
  float best;
  int idx, bad;
  __device__ __forceinline__ void begin() {
    best = -INFINITY;
    idx = INT_MAX;
    bad = 0;
  }
  // The vectors i = tid, tid + kCons, ... < cnt of one ring stage (vector
  // index c0 + i). They arrive in increasing index order per thread, so a
  // strict '>' keeps the first occurrence of the maximum.
  __device__ __forceinline__ void chunk(const uint4* buf, int cnt, int c0, int tid) {
    constexpr int kPer = kChunk / 16 / kCons;
    uint4 v[kPer];
    float vm[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      vm[k] = -INFINITY;
      if (tid + k * kCons < cnt) {
        v[k] = buf[tid + k * kCons];
        vm[k] = E::vmax(v[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (tid + k * kCons < cnt) {
        if (vm[k] != vm[k]) {
          bad = 1;
        } else if (vm[k] > best || idx == INT_MAX) {
          float z[E::kVec];
          E::unpack(v[k], z);
          int j = 0;
#pragma unroll
          for (int jj = E::kVec - 1; jj >= 0; --jj)
            if (z[jj] == vm[k]) j = jj;
          best = vm[k];
          idx = (c0 + tid + k * kCons) * E::kVec + j;
        }
      }
    }
  }
  __device__ void end_row(const Smem& L, int r) {
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
      L.wM[r * kCW + warp] = best;
      L.wI[r * kCW + warp] = anybad ? -2 : idx;
    }
  }
};

// CTA (value, index) of rows [0, nrows) into out[2r], out[2r+1].
__device__ void argmax_to_global(const Smem& L, int nrows, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < nrows; r += kCW) {
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
      out[2 * r] = best;
      out[2 * r + 1] = __int_as_float(bad ? -2 : idx);
    }
  }
}

// Row argmax (-1 for a NaN row) from the S slice partials at float offset 2r.
__device__ int argmax_combine(const GreedyArgs& a, int b, int r) {
  float best = -INFINITY;
  int idx = INT_MAX, bad = 0;
  for (int s = 0; s < a.S; ++s) {
    const float* p = a.ws.part(b, s) + 2 * r;
    const float v = ld_cg_f(p);
    const int i = __float_as_int(ld_cg_f(p + 1));
    if (i == -2) {
      bad = 1;
      continue;
    }
    if (better(v, i, best, idx)) {
      best = v;
      idx = i;
    }
  }
  return (bad || idx == INT_MAX) ? -1 : idx;
}

__device__ bool arrive_row(const GreedyArgs& a, Misc& ms, int b) {
  __threadfence();
  consumers_sync();
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(&a.ws.row_cnt()[b], 1u);
    const int last = (old == uint32_t(a.S) - 1);
    if (last) {
      a.ws.row_cnt()[b] = 0;
      __threadfence();
    }
    ms.last = last;
  }
  consumers_sync();
  return ms.last != 0;
}

__device__ void write_row(const GreedyArgs& a, const Misc& ms, int b, int n, int token, bool error) {
  const int K = a.K;
  for (int i = threadIdx.x; i <= K; i += kCons) {
    int32_t v;
    if (error) v = -1;
    else if (i < n) v = ms.tok[i];
    else if (i == n) v = token;
    else v = -1;
    a.out_tokens[size_t(b) * (K + 1) + i] = v;
  }
  if (threadIdx.x == 0) {
    a.out_n[b] = error ? -1 : n;
    if (error && a.err) atomicOr(a.err, ms.bad_token ? SPEC_DERR_TOKEN : SPEC_DERR_LOGITS);
  }
  __threadfence();
  consumers_sync();
  if (threadIdx.x == 0) atomicAdd(&a.ws.hdr()->rows_done, 1u);
}

template <class E>
__global__ void __launch_bounds__(kThreads, 2) verify_greedy_kernel(const GreedyArgs a) {
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K;
  const Smem L = make_smem(smem_raw, K + 1);
  Misc& ms = *L.misc;
  ring_init(L.ring);
  __syncthreads();
  if (threadIdx.x >= kCons) {
    if (threadIdx.x == kCons) {
      uint32_t it = 0, nt = 0;
      uint64_t idle_t0 = 0;
      int64_t pending = -1;
      WsHeader* h = a.ws.hdr();
      while (!*L.ring.abort && !ld_volatile_u32(&h->abort)) {
        QTask t;
        bool exhausted;
        if (!fetch_task(a.ws, kG1, t, exhausted, pending)) {
          if (!producer_idle(a.ws, exhausted, idle_t0)) break;
          continue;
        }
        idle_t0 = 0;
        const T* tgt = static_cast<const T*>(a.target) + size_t(t.b) * (K + 1) * a.V;
        int v0, v1;
        slice_range(a.nvec, a.S, t.s, v0, v1);
        const char* rows[kMaxK + 1];
        int nrows = 0;
        if (t.type == kG1) {
          for (int i = 0; i < K; ++i) rows[nrows++] = reinterpret_cast<const char*>(tgt + size_t(i) * a.V);
        } else {
          rows[nrows++] = reinterpret_cast<const char*>(tgt + size_t(K) * a.V);
        }
        if (!produce_task(L.ring, it, nt, t, rows, nrows, false, v0, v1)) break;
      }
      produce_end(L.ring, it);
    }
  } else {
    uint32_t it = 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    while (true) {
      if (!wait_stage(L.ring, it)) break;
      const ChunkMeta m0 = L.ring.meta[it % kStages];
      if (m0.slot < 0) break;
      const QTask t = L.ring.ttab[m0.slot];
      const int b = t.b, s = t.s;
      ArgmaxOp<E> op;
      op.begin();
      for (;;) {
        const ChunkMeta m = L.ring.meta[it % kStages];
        const uint4* buf = stage_data(L.ring, it);
        op.chunk(buf, m.c1 - m.c0, m.c0, tid);
        release_stage(L.ring, it);
        ++it;
        if (m.last_k) {
          op.end_row(L, m.r);
          op.begin();
        }
        if (m.last) break;
        if (!wait_stage(L.ring, it)) break;
      }
      consumers_sync();
      const int nrows = (t.type == kG1) ? K : 1;
      argmax_to_global(L, nrows, a.ws.part(b, s));
      if (arrive_row(a, ms, b)) {
        if (warp == 1) {
          int bad = 0;
          if (lane < K) {
            const int d = a.tokens[size_t(b) * K + lane];
            ms.tok[lane] = d;
            bad = (d < 0 || d >= a.V);
          }
          bad = __any_sync(0xffffffffu, bad);
          if (lane == 0) ms.bad_token = bad;
        }
        if (t.type == kG1) {
          for (int r = tid; r < K; r += kCons) ms.best[r] = argmax_combine(a, b, r);
          consumers_sync();
          if (warp == 0) {
            const int g = lane < K ? ms.best[lane] : 0;
            const unsigned mism = __ballot_sync(0xffffffffu, lane < K && g != ms.tok[lane]);
            if (lane == 0) ms.first_mismatch = mism ? (__ffs(int(mism)) - 1) : K;
          }
          consumers_sync();
          const int n = ms.first_mismatch;
          bool error = ms.bad_token != 0;
          for (int i = 0; i <= min(n, K - 1); ++i)
            if (ms.best[i] < 0) error = true;  // a NaN row up to the first mismatch
          if (error || n < K) {
            write_row(a, ms, b, n, error ? -1 : ms.best[n], error);
          } else if (tid == 0) {
            enqueue_row_stage(a.ws, kGB, b, a.S, K);
          }
        } else {
          if (tid == 0) ms.best[K] = argmax_combine(a, b, 0);
          consumers_sync();
          const int tok = ms.best[K];
          write_row(a, ms, b, K, tok, tok < 0 || ms.bad_token != 0);
        }
      }
      consumers_sync();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && (*L.ring.abort || ld_volatile_u32(&a.ws.hdr()->abort))) {
    atomicExch(&a.ws.hdr()->abort, 1u);
    if (a.err) atomicOr(a.err, SPEC_DERR_TIMEOUT);
  }
}

WsLayout greedy_layout(int B, int K, int V, int dtype) {
  const int kvec = (dtype == SPEC_BF16) ? 8 : 4;
  const int nvec = V / kvec;
  return ws_layout(B, slices_for(nvec, B), 2 * K + 2, 1, 2);
}

}  // namespace

size_t greedy_workspace_bytes(int B, int K, int V, int dtype) {
  return greedy_layout(B, K, V, dtype).total;
}

int launch_verify_greedy(const GreedyLaunch& g) {
  GreedyArgs a;
  a.target = g.target;
  a.tokens = g.tokens;
  a.B = g.B;
  a.K = g.K;
  a.V = g.V;
  const int kvec = (g.dtype == SPEC_BF16) ? 8 : 4;
  a.nvec = g.V / kvec;
  const WsLayout wl = greedy_layout(g.B, g.K, g.V, g.dtype);
  a.S = wl.S;
  a.ws.base = static_cast<uint8_t*>(g.workspace);
  a.ws.L = wl;
  a.out_tokens = g.out_tokens;
  a.out_n = g.out_n;
  a.err = g.err;
  cudaStream_t st = static_cast<cudaStream_t>(g.stream);
  if (cudaMemsetAsync(g.workspace, 0, wl.zero_bytes, st) != cudaSuccess) return SPEC_ECUDA;
  const size_t smem = greedy_smem_bytes(g.K + 1);
  if (g.dtype == SPEC_BF16) return launch_dataflow(verify_greedy_kernel<EBf16>, a, smem, st);
  return launch_dataflow(verify_greedy_kernel<EF32>, a, smem, st);
}

}  // namespace sv
