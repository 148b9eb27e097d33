// Paged KV-cache commit/rollback of the accepted provisional slots.
//
// Method: "aiengineeringfromscratch.com - Speculative decoding and EAGLE-3",
// "Rolling back the KV cache" (drafts are written to a scratch area and
// committed on acceptance; rollback costs bytes per layer per head) and
// "Step 4: KV rollback accounting" (new logical length prefix + j + 1);
// "sglang_spec_decode" README, provisional layer (provisional blocks are freed
// at once; no block leaked or freed twice).
//
// Three launches on the caller's stream:
//   kv_plan_kernel   one CTA: validates every row (all-or-nothing), pops the
//                    new tail blocks from the free stack (rows ascending),
//                    then pushes every provisional block (rows ascending) and
//                    writes the call's status word;
//   kv_copy_kernel   one CTA per (row, position <= K): if the status is 0,
//                    copies kept slot s <= n of the row's provisional blocks (slots 0..n,
//                    or slot_map[b][0..n] for a tree draft, whose kept path
//                    need not be contiguous: thakicloud.com, "Speculative
//                    decoding: when it loses", "Grading every branch in one
//                    pass"), for every layer and both K and V planes, to
//                    logical positions L..L+n;
//   kv_finish_kernel one thread per row: sets the new length and clears the
//                    provisional entries. It starts once every copy CTA has
//                    read the tables (programmatic dependent launch), runs
//                    beside the copies and ends by waiting for them, so that
//                    work after it on the stream sees them.
// Only the accepted bytes move: 2 * (n + 1) * layers * heads * head_dim * elem
// bytes read and written per row.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/specverify.h"
#include "launch.h"
#include "launch_util.cuh"
#include "ptx.cuh"

namespace sv {

constexpr int kPlanThreads = 1024;
constexpr int kCopyThreads = 256;

struct KvArgs {
  int32_t* bt;
  int32_t* sl;
  const int32_t* na;
  int32_t* pb;
  uint8_t* pool;
  int NB, NL, H, D, eb, bs;
  int B, K, MB, P;
  int32_t* fs;
  int32_t* ftop;
  int32_t* status;
  const int32_t* smap;  // [B, K + 1] or null (identity)
  int64_t slot_bytes;   // H * D * eb
};

// Provisional slot that kept position s of row b is copied from.
__device__ __forceinline__ int kept_slot(const KvArgs& a, int b, int s) {
  return a.smap ? a.smap[size_t(b) * (a.K + 1) + s] : s;
}

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Adds v (ors when `bits`) into a shared word: one atomic per warp (the warp
// reduces first), not one per thread, which would serialise on the word.
__device__ __forceinline__ void block_add(int* word, int v, bool bits = false) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int y = __shfl_xor_sync(0xffffffffu, v, o);
    v = bits ? (v | y) : (v + y);
  }
  if ((threadIdx.x & 31) == 0 && v != 0) {
    if (bits) atomicOr(word, v);
    else atomicAdd(word, v);
  }
}

// Block-wide exclusive scan of one int per thread (kPlanThreads threads).
__device__ int block_excl_scan(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < kPlanThreads / 32 ? sh[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    sh[32 + lane] = wi - w;
    if (lane == 31) sh[64] = wi;
  }
  __syncthreads();
  const int res = sh[32 + warp] + inc - v;
  total = sh[64];
  __syncthreads();
  return res;
}

// Validation of one row; returns error bits, the number of new blocks and of
// provisional blocks to push.
__device__ int validate_row(const KvArgs& a, int b, int& need, int& npush) {
  int e = 0;
  need = 0;
  npush = 0;
  const int n = a.na[b], L = a.sl[b];
  for (int k = 0; k < a.P; ++k) {
    const int x = a.pb[size_t(b) * a.P + k];
    if (x >= 0) {
      ++npush;
      if (x >= a.NB) e |= SPEC_DERR_BAD_BLOCK;
    }
  }
  if (n < 0 || n > a.K) return e | SPEC_DERR_BAD_ACCEPT;
  if (L < 0 || cdiv(L + n + 1, a.bs) > a.MB) return e | SPEC_DERR_BAD_LENGTH;
  const int have = cdiv(L, a.bs), tot = cdiv(L + n + 1, a.bs);
  for (int j = L / a.bs; j < tot; ++j) {
    const int x = a.bt[size_t(b) * a.MB + j];
    if (j < have) {
      if (x < 0 || x >= a.NB) e |= SPEC_DERR_BAD_BLOCK;  // the partly filled tail block
    } else if (x != -1) {
      e |= SPEC_DERR_BAD_BLOCK;  // a slot the commit must fill is already taken
    }
  }
  int slot_err = 0, blk_err = 0;
  for (int s = 0; s <= n; ++s) {  // the provisional blocks of the kept slots
    const int x = kept_slot(a, b, s);
    if (x < 0 || x > a.K) {
      slot_err = 1;
    } else if (x / a.bs >= a.P) {
      blk_err = 1;
    } else {
      const int y = a.pb[size_t(b) * a.P + x / a.bs];
      if (y < 0 || y >= a.NB) blk_err = 1;
    }
  }
  if (slot_err) e |= SPEC_DERR_BAD_SLOT;
  else if (blk_err) e |= SPEC_DERR_BAD_BLOCK;
  need = tot - have;
  return e;
}

__global__ void __launch_bounds__(kPlanThreads) kv_plan_kernel(const KvArgs a) {
  __shared__ int sh[96];
  __shared__ int s_err, s_need, s_push;
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // the verification that produced num_accepted
  if (tid == 0) {
    s_err = 0;
    s_need = 0;
    s_push = 0;
  }
  __syncthreads();
  // 1. validation and totals; with one row per thread (B <= kPlanThreads) the
  // row's counts stay in registers for the pops and pushes below
  const bool one = a.B <= kPlanThreads;
  int e = 0, need_sum = 0, push_sum = 0, my_need = 0, my_np = 0;
  for (int b = tid; b < a.B; b += kPlanThreads) {
    int need, np;
    e |= validate_row(a, b, need, np);
    need_sum += need;
    push_sum += np;
    my_need = need;
    my_np = np;
  }
  block_add(&s_err, e, true);
  block_add(&s_need, need_sum);
  block_add(&s_push, push_sum);
  __syncthreads();
  const int top = *a.ftop;
  int err = s_err;
  const int need_total = s_need, push_total = s_push;
  if (err == 0 && (top < 0 || top > a.NB || need_total > top)) err |= SPEC_DERR_NO_SPACE;
  if (err == 0 && top - need_total + push_total > a.NB) err |= SPEC_DERR_BAD_BLOCK;
  if (err == 0) {
    // every block about to be popped must be a valid id
    int pe = 0;
    for (int i = top - need_total + tid; i < top; i += kPlanThreads) {
      const int x = a.fs[i];
      if (x < 0 || x >= a.NB) pe = 1;
    }
    block_add(&s_err, pe ? SPEC_DERR_BAD_BLOCK : 0, true);
    __syncthreads();
    err |= s_err;
  }
  if (err != 0) {
    if (tid == 0) *a.status = err;
    return;
  }
  // 2. pops: row b takes free_stack[top-1-(prefix_b+k)], rows ascending
  int carry = 0;
  for (int b0 = 0; b0 < a.B; b0 += kPlanThreads) {
    const int b = b0 + tid;
    int need = my_need, np = 0;
    if (!one) {
      need = 0;
      if (b < a.B) validate_row(a, b, need, np);
    }
    int chunk_total;
    const int pre = block_excl_scan(need, sh, chunk_total) + carry;
    if (b < a.B) {
      const int have = cdiv(a.sl[b], a.bs);
      for (int k = 0; k < need; ++k)
        a.bt[size_t(b) * a.MB + have + k] = a.fs[top - 1 - (pre + k)];
    }
    carry += chunk_total;
  }
  __syncthreads();  // all pops have read the stack before any push writes it
  // 3. pushes: provisional blocks, rows ascending, from the new top
  const int base = top - need_total;
  carry = 0;
  for (int b0 = 0; b0 < a.B; b0 += kPlanThreads) {
    const int b = b0 + tid;
    int np = my_np;
    if (!one) {
      np = 0;
      if (b < a.B)
        for (int k = 0; k < a.P; ++k) np += a.pb[size_t(b) * a.P + k] >= 0;
    }
    int chunk_total;
    const int pre = block_excl_scan(np, sh, chunk_total) + carry;
    if (b < a.B) {
      int w = 0;
      for (int k = 0; k < a.P; ++k) {
        const int x = a.pb[size_t(b) * a.P + k];
        if (x >= 0) a.fs[base + pre + (w++)] = x;
      }
    }
    carry += chunk_total;
  }
  if (tid == 0) {
    *a.ftop = base + push_total;
    *a.status = 0;
  }
}

__global__ void __launch_bounds__(kCopyThreads) kv_copy_kernel(const KvArgs a) {
  // one CTA per (row, kept position): every SM takes a share of the slots,
  // whatever the rows' accepted lengths
  const int b = blockIdx.x / (a.K + 1), s = blockIdx.x % (a.K + 1);
  pdl_wait();  // the plan
  if (*a.status != 0) return;
  const int n = a.na[b];
  if (s > n) return;
  const int L = a.sl[b];
  const int64_t layer_stride = int64_t(2) * a.bs * a.slot_bytes;  // one layer: K and V planes
  const int64_t block_stride = int64_t(a.NL) * layer_stride;
  const int x = kept_slot(a, b, s);
  const int sb = a.pb[size_t(b) * a.P + x / a.bs];
  const int pos = L + s;
  const int db = a.bt[size_t(b) * a.MB + pos / a.bs];
  const uint8_t* src = a.pool + int64_t(sb) * block_stride + int64_t(x % a.bs) * a.slot_bytes;
  uint8_t* dst = a.pool + int64_t(db) * block_stride + int64_t(pos % a.bs) * a.slot_bytes;
  // A barrier that takes the read values as operands: every table read of
  // the CTA has returned before the trigger lets the finish change the
  // tables. (The plan validated these ids; the test cannot fail.)
  if (__syncthreads_or(sb < 0 || db < 0 || L < 0 || x < 0)) return;
  pdl_trigger();
  const int vpu = int(a.slot_bytes / 16);  // 16-byte vectors per (layer, plane)
  const int total = 2 * a.NL * vpu;
  const int64_t plane_stride = int64_t(a.bs) * a.slot_bytes;
  constexpr int kUnroll = 8;
  for (int g0 = threadIdx.x; g0 < total; g0 += kCopyThreads * kUnroll) {
    uint4 v[kUnroll];
    int64_t off[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      const int g = g0 + i * kCopyThreads;
      off[i] = -1;
      if (g < total) {
        const int u = g / vpu;  // layer * 2 + plane
        off[i] = int64_t(u) * plane_stride + int64_t(g - u * vpu) * 16;
        v[i] = ldg_nc_v4(src + off[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < kUnroll; ++i)
      if (off[i] >= 0) *reinterpret_cast<uint4*>(dst + off[i]) = v[i];
  }
}

// The new lengths and the cleared provisional entries (the copy CTAs read
// both, so they change only once every copy CTA has read them).
__global__ void __launch_bounds__(256) kv_finish_kernel(const KvArgs a) {
  const int b = blockIdx.x * 256 + threadIdx.x;
  // every copy CTA has read the tables (they trigger after their reads); the
  // plan, which they waited for, is complete
  if (b < a.B && *a.status == 0) {
    a.sl[b] = a.sl[b] + a.na[b] + 1;
    for (int i = 0; i < a.P; ++i) a.pb[size_t(b) * a.P + i] = -1;
  }
  pdl_wait();  // every copy: work after this launch on the stream sees them
}

// ------------------------------------------------------------------ in place
// The in-place variant ("Rolling back the KV cache": keep the physical cache
// and truncate a logical length; the sglang_spec_decode README: evict a row's
// provisional KV on preemption). The K+1 provisional slots already sit at
// logical positions L..L+K of the row's own blocks; the new length is
// L + n + 1 (commit) or L (evict), and every block holding no position below
// it is pushed onto the free stack (rows ascending, block index ascending)
// and cleared in the block table. No KV byte moves. One CTA, all-or-nothing.
struct TruncArgs {
  int32_t* bt;
  int32_t* sl;
  const int32_t* na;  // null: evict
  int NB, bs, B, K, MB;
  int32_t* fs;
  int32_t* ftop;
  int32_t* status;
};

// Validation of one row; returns error bits, the new length and the block
// range [first, end) to free.
__device__ int validate_trunc_row(const TruncArgs& a, int b, int& new_len, int& first, int& end) {
  new_len = first = end = 0;
  const int L = a.sl[b];
  const int n = a.na ? a.na[b] : 0;
  if (a.na && (n < 0 || n > a.K)) return SPEC_DERR_BAD_ACCEPT;
  if (L < 0 || int64_t(L) + a.K + 1 > int64_t(a.MB) * a.bs) return SPEC_DERR_BAD_LENGTH;
  end = cdiv(L + a.K + 1, a.bs);
  int e = 0;
  for (int j = L / a.bs; j < end; ++j) {
    const int x = a.bt[size_t(b) * a.MB + j];
    if (x < 0 || x >= a.NB) e |= SPEC_DERR_BAD_BLOCK;
  }
  new_len = a.na ? L + n + 1 : L;
  first = cdiv(new_len, a.bs);
  return e;
}

__global__ void __launch_bounds__(kPlanThreads) kv_truncate_kernel(const TruncArgs a) {
  __shared__ int sh[96];
  __shared__ int s_err, s_push;
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // the verification that produced num_accepted
  if (tid == 0) {
    s_err = 0;
    s_push = 0;
  }
  __syncthreads();
  int e = 0, push_sum = 0;
  for (int b = tid; b < a.B; b += kPlanThreads) {
    int nl, f, en;
    e |= validate_trunc_row(a, b, nl, f, en);
    push_sum += en - f;
  }
  block_add(&s_err, e, true);
  block_add(&s_push, push_sum);
  __syncthreads();
  const int top = *a.ftop;
  int err = s_err;
  if (err == 0 && (top < 0 || top + s_push > a.NB)) err |= SPEC_DERR_BAD_BLOCK;
  if (err != 0) {
    if (tid == 0) *a.status = err;
    return;
  }
  int carry = 0;
  for (int b0 = 0; b0 < a.B; b0 += kPlanThreads) {
    const int b = b0 + tid;
    int nl = 0, f = 0, en = 0;
    if (b < a.B) validate_trunc_row(a, b, nl, f, en);
    int chunk_total;
    const int pre = block_excl_scan(en - f, sh, chunk_total) + carry;
    if (b < a.B) {
      for (int j = f; j < en; ++j) {
        int32_t* slot = &a.bt[size_t(b) * a.MB + j];
        a.fs[top + pre + (j - f)] = *slot;
        *slot = -1;
      }
      a.sl[b] = nl;
    }
    carry += chunk_total;
  }
  if (tid == 0) {
    *a.ftop = top + s_push;
    *a.status = 0;
  }
}

int launch_kv_truncate(const KvTruncLaunch& k) {
  TruncArgs a{k.block_table, k.seq_lens, k.num_accepted, k.num_blocks, k.block_size, k.B, k.K,
              k.max_blocks, k.free_stack, k.free_top, k.status};
  return launch_pdl(kv_truncate_kernel, dim3(1), dim3(kPlanThreads), 0,
                    static_cast<cudaStream_t>(k.stream), a);
}

int launch_kv_commit(const KvLaunch& k) {
  KvArgs a;
  a.bt = k.block_table;
  a.sl = k.seq_lens;
  a.na = k.num_accepted;
  a.pb = k.prov_blocks;
  a.pool = static_cast<uint8_t*>(k.kv_pool);
  a.NB = k.num_blocks;
  a.NL = k.num_layers;
  a.H = k.num_kv_heads;
  a.D = k.head_dim;
  a.eb = k.elem_bytes;
  a.bs = k.block_size;
  a.B = k.B;
  a.K = k.K;
  a.MB = k.max_blocks;
  a.P = k.P;
  a.fs = k.free_stack;
  a.ftop = k.free_top;
  a.status = k.status;
  a.smap = k.slot_map;
  a.slot_bytes = int64_t(k.num_kv_heads) * k.head_dim * k.elem_bytes;
  cudaStream_t st = static_cast<cudaStream_t>(k.stream);
  // each launch starts while its predecessor finishes and waits for it
  // (programmatic dependent launch), so the three hide each other's launch gaps
  if (launch_pdl(kv_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, a) != SPEC_OK)
    return SPEC_ECUDA;
  if (launch_pdl(kv_copy_kernel, dim3(k.B * (k.K + 1)), dim3(kCopyThreads), 0, st, a) != SPEC_OK)
    return SPEC_ECUDA;
  return launch_pdl(kv_finish_kernel, dim3((k.B + 255) / 256), dim3(256), 0, st, a);
}

}  // namespace sv
