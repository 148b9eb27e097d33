// Greedy verification kernel (spec_verify_greedy).
//
// Method ("devpost.com - phoenix", "What it does"): tokens are kept up to the
// first disagreement between the draft token and the target's argmax, where
// the target's own token is written; the output equals the target decoding
// alone. Ties in the argmax go to the lowest vocabulary index.
//
// GB300 mapping (dataflow engine, engine.cuh): task (b, s) streams slice s of
// target rows 0..K-1; the consumer warps leave per-warp (max, first index)
// pairs in a hand-off slot, the finisher warp combines them into the slice's
// partials and arrives on the row's counter. The finisher completing row b
// combines the S partials, finds the first mismatch with a warp ballot, and
// either writes the row or (all K accepted) enqueues the slices of target row
// K, whose completing finisher writes the bonus token. Raw logits are compared
// exactly (no temperature).
//
// Tree mode (spec_verify_tree_greedy; thakicloud.com, "Speculative decoding:
// when it loses", section "Grading every branch in one pass": the
// flattened draft tree is graded in one target pass and the longest surviving
// path is kept): N nodes in topological order, target row 0 after the
// committed prefix and row 1 + i after node i. The single stage streams all
// N + 1 rows; the finisher that completes a row keeps the deepest node whose
// whole root path matches the target's argmaxes and emits the path, then the
// argmax of its last node's row. With distinct sibling tokens this equals
// target-only greedy decoding, as in the linear case.
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
constexpr int kFinWarp = kCW + 1;  // warp index of the finisher

struct GreedyArgs {
  const void* target;
  const int32_t* tokens;
  int B, K, V, S, nvec;  // tree mode: K = N nodes
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  const int32_t* parents;  // tree mode: [B, N] parent of each node (-1: root); else null
  int32_t* out_slots;      // tree mode, optional: [B, N + 1] KV slot of each kept position
  unsigned long long* counters;  // optional acceptance statistics [2K + 2]
  Ws ws;
};

// Hand-off slot: the task (16 bytes), then float wM[R][kCW], int wI[R][kCW]
// (index -2: a NaN was seen); R = rows a first-stage task reads.
__host__ __device__ inline int slot_bytes(int R) { return (16 + R * kCW * 8 + 15) / 16 * 16; }

struct Smem {
  Ring ring;
  Handoff ho;
  float2* item;  // [256] finisher scratch: slice partials being combined
};

__host__ __device__ inline size_t greedy_smem_bytes(int R) {
  size_t o = size_t(kStages) * kChunk;
  o += 2 * kStages * 8;
  o += kStages * sizeof(ChunkMeta) + kStages * sizeof(QTask);
  o += 2 * kSlots * 8 + 16;
  o += 256 * 8;
  o += size_t(kSlots) * slot_bytes(R);
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
  L.ho.done = reinterpret_cast<uint64_t*>(base + o);
  L.ho.freed = L.ho.done + kSlots;
  o += 2 * kSlots * 8;
  L.ring.abort = reinterpret_cast<volatile int*>(base + o);
  o += 16;
  L.item = reinterpret_cast<float2*>(base + o);
  o += 256 * 8;
  L.ho.data = base + o;
  L.ho.slot_bytes = slot_bytes(R);
  return L;
}

// Target rows a first-stage task reads: 0..K-1, or 0..N in tree mode.
__device__ __host__ __forceinline__ int rows_of(const GreedyArgs& a) {
  return a.parents ? a.K + 1 : a.K;
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
  // Warp partial of row r into the hand-off slot.
  __device__ __forceinline__ void end_row(uint8_t* slot, int R, int r) {
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
      float* wM = reinterpret_cast<float*>(slot + 16);
      int* wI = reinterpret_cast<int*>(wM + R * kCW);
      wM[r * kCW + warp] = best;
      wI[r * kCW + warp] = anybad ? -2 : idx;
    }
  }
};

// Finisher: slice partial (value, index) of the task's rows into out[2r], out[2r+1].
__device__ void combine_task(const GreedyArgs& a, const QTask& t, const uint8_t* slot) {
  const int lane = threadIdx.x & 31;
  const int R = rows_of(a), nrows = (t.type == kG1) ? rows_of(a) : 1;
  const float* wM = reinterpret_cast<const float*>(slot + 16);
  const int* wI = reinterpret_cast<const int*>(wM + R * kCW);
  float* out = a.ws.part(t.b, t.s);
  for (int r = lane; r < nrows; r += 32) {
    float best = -INFINITY;
    int idx = INT_MAX, bad = 0;
#pragma unroll
    for (int q = 0; q < kCW; ++q) {
      const float v = wM[r * kCW + q];
      const int i = wI[r * kCW + q];
      if (i == -2) bad = 1;
      else if (better(v, i, best, idx)) {
        best = v;
        idx = i;
      }
    }
    out[2 * r] = best;
    out[2 * r + 1] = __int_as_float(bad ? -2 : idx);
  }
  __syncwarp();
}

// Row argmax (-1 for a NaN row) of rows [0, nrows) from the S slice
// partials (float offset 2r: value, index or -2 for NaN); the partials of a
// group of rows are loaded by all lanes at once, then lane r combines row r.
// The result of row r ends in lane r (r < 32).
__device__ int argmax_rows(const GreedyArgs& a, const Smem& L, int b, int nrows) {
  const int lane = threadIdx.x & 31, S = a.S;
  const int per_group = 256 / S > 0 ? 256 / S : 1;
  int res = -1;
  for (int r0 = 0; r0 < nrows; r0 += per_group) {
    const int rg = min(per_group, nrows - r0), items = rg * S;
#pragma unroll 8
    for (int i = lane; i < items; i += 32) {
      const int r = r0 + i / S, sl = i % S;
      L.item[i] = __ldcg(reinterpret_cast<const float2*>(a.ws.part(b, sl) + 2 * r));
    }
    __syncwarp();
    for (int rr = lane - r0; rr >= 0 && rr < rg; rr += 32) {
      float best = -INFINITY;
      int idx = INT_MAX, bad = 0;
      for (int sl = 0; sl < S; ++sl) {
        const float2 v = L.item[rr * S + sl];
        const int i = __float_as_int(v.y);
        if (i == -2) bad = 1;
        else if (better(v.x, i, best, idx)) {
          best = v.x;
          idx = i;
        }
      }
      res = (bad || idx == INT_MAX) ? -1 : idx;
    }
    __syncwarp();
  }
  return res;
}

__device__ void write_row(const GreedyArgs& a, int b, int n, int token, bool error, int errbits) {
  const int lane = threadIdx.x & 31, K = a.K;
  for (int i = lane; i <= K; i += 32) {
    int32_t v;
    if (error) v = -1;
    else if (i < n) v = a.tokens[size_t(b) * K + i];
    else if (i == n) v = token;
    else v = -1;
    a.out_tokens[size_t(b) * (K + 1) + i] = v;
  }
  if (lane == 0) {
    a.out_n[b] = error ? -1 : n;
    if (error && a.err) atomicOr(a.err, errbits);
    atomicAdd(&a.ws.hdr()->rows_done, 1u);  // lets the producers stop; no ordering needed
  }
  if (a.counters && !error) count_acceptance(a.counters, K, n);
  __syncwarp();
}

// G1 complete: first mismatch between draft tokens and the target argmaxes.
__device__ void finish_g1(const GreedyArgs& a, const Smem& L, int b) {
  const int lane = threadIdx.x & 31, K = a.K;
  int d = 0, badtok = 0;
  if (lane < K) {
    d = a.tokens[size_t(b) * K + lane];
    badtok = (d < 0 || d >= a.V);
  }
  const int g = argmax_rows(a, L, b, K);
  badtok = __any_sync(0xffffffffu, badtok);
  const unsigned mism = __ballot_sync(0xffffffffu, lane < K && g != d);
  const int n = mism ? (__ffs(int(mism)) - 1) : K;
  // a NaN row up to the first mismatch is an error
  const int nan_row = __any_sync(0xffffffffu, lane < K && lane <= n && g < 0);
  if (badtok || nan_row) {
    write_row(a, b, n, -1, true, badtok ? SPEC_DERR_TOKEN : SPEC_DERR_LOGITS);
    return;
  }
  if (n < K) {
    write_row(a, b, n, __shfl_sync(0xffffffffu, g, n), false, 0);
    return;
  }
  enqueue_row_stage(a.ws, kGB, b, a.S, K);
}

// GB complete: the bonus token is the argmax of target row K.
__device__ void finish_gb(const GreedyArgs& a, const Smem& L, int b) {
  const int tok = __shfl_sync(0xffffffffu, argmax_rows(a, L, b, 1), 0);
  write_row(a, b, a.K, tok, tok < 0, SPEC_DERR_LOGITS);
}

// Tree mode. Lane i holds node i (parent, token) and the argmax of row i.
// Node i is consistent when its token is the argmax of its parent's row; it
// survives when every node on its root path is consistent. Pointer jumping
// (five rounds cover depth 31) gives each node its survival and depth at
// once; the kept path ends at the deepest survivor, the lowest index among
// equally deep ones, and is read back by walking its parents.
__device__ void finish_tree(const GreedyArgs& a, const Smem& L, int b) {
  const int lane = threadIdx.x & 31, N = a.K;
  int par = -1, tok = -1, bad = 0;
  if (lane < N) {
    par = a.parents[size_t(b) * N + lane];
    tok = a.tokens[size_t(b) * N + lane];
    bad = tok < 0 || tok >= a.V || par < -1 || par >= lane;
  }
  const int g = argmax_rows(a, L, b, N + 1);  // lane r: argmax of row r, -1 if unusable
  bad = __any_sync(0xffffffffu, bad);
  if (bad) par = -1;  // keeps the shuffles below in range
  const int g_par = __shfl_sync(0xffffffffu, g, par + 1);
  int alive = lane < N && g_par >= 0 && tok == g_par;
  int depth = 1, anc = par;
#pragma unroll
  for (int round = 0; round < 5; ++round) {
    const int src = anc >= 0 ? anc : lane;
    const int a_alive = __shfl_sync(0xffffffffu, alive, src);
    const int a_depth = __shfl_sync(0xffffffffu, depth, src);
    const int a_anc = __shfl_sync(0xffffffffu, anc, src);
    if (anc >= 0) {
      alive &= a_alive;
      depth += a_depth;
      anc = a_anc;
    }
  }
  alive = alive && lane < N;
  const int g_own = __shfl_sync(0xffffffffu, g, min(lane + 1, 31));
  const bool error = bad || __shfl_sync(0xffffffffu, g, 0) < 0 ||
                     __any_sync(0xffffffffu, alive && g_own < 0);
  const int key = __reduce_max_sync(0xffffffffu, alive ? (depth << 8) | (255 - lane) : -1);
  const int best = key < 0 ? -1 : 255 - (key & 255);
  const int n = key < 0 ? 0 : key >> 8;
  int my_node = -1;  // lane p: the node at depth p + 1 of the kept path
  for (int cur = best; cur >= 0;) {
    if (lane == __shfl_sync(0xffffffffu, depth, cur) - 1) my_node = cur;
    cur = __shfl_sync(0xffffffffu, par, cur);
  }
  const int node_tok = __shfl_sync(0xffffffffu, tok, my_node < 0 ? 0 : my_node);
  const int prev_node = __shfl_up_sync(0xffffffffu, my_node, 1);
  const int last = __shfl_sync(0xffffffffu, g, best + 1);
  if (lane <= N) {
    int32_t v = -1, sl = -1;
    if (!error) {
      if (lane < n) v = node_tok;
      if (lane == n) v = last;
      // kept position p: slot 0 (last committed token) or 1 + the node at depth p
      if (lane <= n) sl = lane == 0 ? 0 : 1 + prev_node;
    }
    a.out_tokens[size_t(b) * (N + 1) + lane] = v;
    if (a.out_slots) a.out_slots[size_t(b) * (N + 1) + lane] = sl;
  }
  if (lane == 0) {
    a.out_n[b] = error ? -1 : n;
    if (error && a.err) atomicOr(a.err, bad ? SPEC_DERR_TOKEN : SPEC_DERR_LOGITS);
    atomicAdd(&a.ws.hdr()->rows_done, 1u);
  }
  __syncwarp();
}

template <class E>
__global__ void __launch_bounds__(kThreads, 2) verify_greedy_kernel(const GreedyArgs a) {
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K, R = rows_of(a);
  const Smem L = make_smem(smem_raw, R);
  ring_init(L.ring);
  handoff_init(L.ho);
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // the workspace zeroing launched just before
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* h = a.ws.hdr();

  if (warp == kCW) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0, nt = 0;
      uint64_t idle_t0 = 0;
      Fetcher fx;
      while (!*L.ring.abort && !ld_volatile_u32(&h->abort)) {
        QTask t;
        if (!fx.next(a.ws, kG1, t)) {
          if (!producer_idle(a.ws, !fx.first_left, idle_t0)) break;
          continue;
        }
        idle_t0 = 0;
        const T* tgt = static_cast<const T*>(a.target) + size_t(t.b) * (K + 1) * a.V;
        int v0, v1;
        slice_range(a.nvec, a.S, t.s, v0, v1);
        // G1: target rows 0..R-1; GB: target row K
        const int nrows = (t.type == kG1) ? R : 1;
        const int r0 = (t.type == kG1) ? 0 : K;
        auto row = [&](int r) { return reinterpret_cast<const char*>(tgt + size_t(r0 + r) * a.V); };
        auto prefetch = [&]() { fx.prepare(a.ws); };
        if (!produce_task(L.ring, it, nt, t, row, nrows, false, v0, v1, prefetch)) break;
      }
      produce_end(L.ring, it);
    }
  } else if (warp == kFinWarp) {
    // ------------------------------------------------ finisher
    finisher_loop(
        a.ws, L.ho, L.ring.abort,
        [&](const QTask& t, const uint8_t* slot) { combine_task(a, t, slot); },
        [&](const QTask& t) {
          if (a.parents) finish_tree(a, L, t.b);
          else if (t.type == kG1) finish_g1(a, L, t.b);
          else finish_gb(a, L, t.b);
        },
        [&](const QTask&) { return a.S; });
  } else {
    // ------------------------------------------------ consumers
    const int tid = threadIdx.x;
    uint32_t it = 0, n = 0;
    for (;; ++n) {
      if (!wait_stage(L.ring, it)) break;
      const ChunkMeta m0 = L.ring.meta[it % kStages];
      if (m0.slot < 0) break;
      const QTask t = L.ring.ttab[m0.slot];
      if (!handoff_acquire(L.ho, n)) {
        *L.ring.abort = 1;
        break;
      }
      uint8_t* slot = L.ho.slot(n);
      if (tid == 0) *reinterpret_cast<QTask*>(slot) = t;
      ArgmaxOp<E> op;
      op.begin();
      bool ok = true;
      for (;;) {
        const ChunkMeta m = L.ring.meta[it % kStages];
        op.chunk(stage_data(L.ring, it), m.c1 - m.c0, m.c0, tid);
        release_stage(L.ring, it);
        ++it;
        if (m.last_k) {
          op.end_row(slot, R, m.r);
          op.begin();
        }
        if (m.last) break;
        if (!wait_stage(L.ring, it)) {
          ok = false;
          break;
        }
      }
      handoff_post(L.ho, n);
      if (!ok) {
        ++n;
        break;
      }
    }
    // end of stream for the finisher
    if (handoff_acquire(L.ho, n)) {
      if (tid == 0) *reinterpret_cast<QTask*>(L.ho.slot(n)) = QTask{0, 0, 0, 0};
      handoff_post(L.ho, n);
    } else {
      *L.ring.abort = 1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && (*L.ring.abort || ld_volatile_u32(&h->abort))) {
    atomicExch(&h->abort, 1u);
    if (a.err) atomicOr(a.err, SPEC_DERR_TIMEOUT);
  }
}

WsLayout greedy_layout(int B, int K, int V, int dtype) {
  const int kvec = (dtype == SPEC_BF16) ? 8 : 4;
  const int nvec = V / kvec;
  return ws_layout(B, slices_for(nvec, B, small_batch(B, small_batch_knob(), kGreedySmallBatch),
                                         kGreedyTasks),
                   2 * K + 2, 1, 2, 16);
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
  set_test_knobs(a.ws);
  a.out_tokens = g.out_tokens;
  a.out_n = g.out_n;
  a.err = g.err;
  a.counters = g.parents ? nullptr : g.counters;
  a.parents = g.parents;
  a.out_slots = g.out_slots;
  cudaStream_t st = static_cast<cudaStream_t>(g.stream);
  if (zero_workspace(g.workspace, wl.zero_bytes, st) != SPEC_OK) return SPEC_ECUDA;
  const size_t smem = greedy_smem_bytes(rows_of(a));
  if (g.dtype == SPEC_BF16) return launch_dataflow(verify_greedy_kernel<EBf16>, a, smem, st);
  return launch_dataflow(verify_greedy_kernel<EF32>, a, smem, st);
}

}  // namespace sv
