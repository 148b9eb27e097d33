// Dataflow engine of the verification kernels.
//
// The batch is cut into tasks: task (b, s) works on vocabulary slice s of
// batch row b. Every kernel is persistent (one or two CTAs per SM, no
// clusters). In each CTA one producer thread fetches tasks and streams their
// logit slices from global memory into a ring of shared-memory stages with
// 1-D bulk async copies (completion on mbarriers); eight consumer warps
// process the stages in order. A task leaves its partial results (per-slice
// sums) in an L2-resident workspace and arrives on an atomic counter of its
// row; the CTA whose arrival completes the row's stage combines the partials
// and continues the row: it decides, writes outputs, or enqueues the row's
// next stage as new tasks. No CTA ever waits for another one, so the HBM
// stream never stalls behind a row's serial steps.
//
// Task sources, in priority order: the dynamic queue (later stages of rows
// already started, which keeps their data hot in L2), then the static list of
// first-stage tasks (b, s) in row order. Every wait is bounded; a timeout sets
// the workspace abort word, the kernel drains, and unfinished rows keep the -1
// outputs the host pre-filled.
#pragma once
#include <cstdint>

#include "../../include/specverify.h"
#include "common.cuh"
#include "ptx.cuh"

namespace sv {

// ------------------------------------------------------------------ slicing
// Vocabulary slices per batch row. At least enough that one row slice fits
// one ring stage (kChunk bytes); for small batches more, up to kTargetTasks
// first-stage tasks so that every persistent CTA gets work (slices of at least
// 64 vectors); never more than kMaxSlices (two warp-wide scans in the draw).
constexpr int kMaxSlices = 64;
constexpr int kTargetTasks = 608;  // two per CTA of a 152-SM GB300 at two CTAs per SM

__host__ __device__ inline int slices_for(int nvec, int B) {
  const int per = kChunk / 16;
  int s = (nvec + per - 1) / per;
  int par = (kTargetTasks + B - 1) / B;
  const int cap = nvec / 64 > 1 ? nvec / 64 : 1;
  if (par > cap) par = cap;
  if (s < par) s = par;
  if (s > kMaxSlices) s = kMaxSlices;
  if (s > nvec) s = nvec;
  return s < 1 ? 1 : s;
}

// ------------------------------------------------------------------ workspace
struct WsHeader {           // zeroed by the host before every launch
  uint32_t p1_next;         // next first-stage task
  uint32_t dq_tail;         // dynamic-queue reservations
  uint32_t dq_head;         // dynamic-queue claims
  uint32_t rows_done;       // rows whose outputs are written
  uint32_t abort;           // set on any timeout
  uint32_t pad[3];
};

struct QTask {
  int type, b, s, aux;
};

// Offsets (bytes) of the workspace regions; computed identically on host and device.
struct WsLayout {
  size_t header, row_cnt, ready, entries, part, units, rowstate, total, zero_bytes;
  int B, S, qcap, part_floats, ustride;
};

// per-row state written by the row's finishers
struct RowState {
  int n, flags, mode, err;  // mode: 0 residual (q_j, p_j), 1 draw from q alone
  float Kq, Kp, Rq, Rp;     // integer offsets and fp32 1/S of the draw's rows
  float Iq_hi, Iq_lo, Ip_hi, Ip_lo;  // accurate 1/S (double-float path)
  float pad[4];
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) / 256 * 256; }

// part_floats: floats of partial results per (row, slice); ustride: unit slots per slice.
__host__ __device__ inline WsLayout ws_layout(int B, int S, int part_floats, int ustride,
                                              int stages_per_row) {
  WsLayout w;
  w.B = B;
  w.S = S;
  w.qcap = B * S * stages_per_row;
  w.part_floats = part_floats;
  w.ustride = ustride;
  size_t o = 0;
  w.header = o;
  o += ws_align(sizeof(WsHeader));
  w.row_cnt = o;
  o += ws_align(size_t(B) * 4);
  w.ready = o;
  o += ws_align(size_t(w.qcap) * 4);
  w.zero_bytes = o;  // everything above is zeroed per call
  w.entries = o;
  o += ws_align(size_t(w.qcap) * sizeof(QTask));
  w.part = o;
  o += ws_align(size_t(B) * S * part_floats * 4);
  w.units = o;
  o += ws_align(size_t(B) * S * ustride * 8);
  w.rowstate = o;
  o += ws_align(size_t(B) * sizeof(RowState));
  w.total = o;
  return w;
}

struct Ws {
  uint8_t* base;
  WsLayout L;
  __device__ WsHeader* hdr() const { return reinterpret_cast<WsHeader*>(base + L.header); }
  __device__ uint32_t* row_cnt() const { return reinterpret_cast<uint32_t*>(base + L.row_cnt); }
  __device__ uint32_t* ready() const { return reinterpret_cast<uint32_t*>(base + L.ready); }
  __device__ QTask* entries() const { return reinterpret_cast<QTask*>(base + L.entries); }
  __device__ float* part(int b, int s) const {
    return reinterpret_cast<float*>(base + L.part) + (size_t(b) * L.S + s) * L.part_floats;
  }
  __device__ float2* units(int b, int s) const {
    return reinterpret_cast<float2*>(base + L.units) + (size_t(b) * L.S + s) * L.ustride;
  }
  __device__ RowState* rowstate(int b) const {
    return reinterpret_cast<RowState*>(base + L.rowstate) + b;
  }
};

// ------------------------------------------------------------------ memory helpers
__device__ __forceinline__ float ld_cg_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ int ld_cg_i(const int* p) { return __ldcg(p); }
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

// ------------------------------------------------------------------ queue
// Appends n tasks (type, b, s = 0..n-1, aux). One calling thread. A queue
// overflow (more later-stage tasks than the layout provides) aborts the launch.
__device__ inline void enqueue_row_stage(const Ws& ws, int type, int b, int n, int aux) {
  const uint32_t base = atomicAdd(&ws.hdr()->dq_tail, uint32_t(n));
  if (base + uint32_t(n) > uint32_t(ws.L.qcap)) {
    atomicExch(&ws.hdr()->abort, 1u);
    return;
  }
  QTask* e = ws.entries();
  for (int s = 0; s < n; ++s) e[base + s] = QTask{type, b, s, aux};
  __threadfence();
  for (int s = 0; s < n; ++s) st_release_u32(&ws.ready()[base + s], 1u);
}

// The producer's fetch. Queued tasks are claimed by ticket: a producer that
// sees the queue non-empty takes the next ticket with one atomicAdd (no
// compare-and-swap retries, which serialise hundreds of producers on one
// word) and from then on polls only that entry's ready flag. A ticket can
// outrun the queue (several producers saw the same last entry); its holder
// keeps taking first-stage tasks until the entry appears, and once every row
// is done the ticket is simply dropped. `pending` is the held ticket (-1:
// none). Returns false when nothing is runnable now; `exhausted` then says
// that no first-stage task is left.
__device__ inline bool fetch_task(const Ws& ws, int first_type, QTask& t, bool& exhausted,
                                  int64_t& pending) {
  WsHeader* h = ws.hdr();
  exhausted = false;
  if (pending < 0) {
    const uint32_t head = ld_volatile_u32(&h->dq_head);
    const uint32_t tail = ld_volatile_u32(&h->dq_tail);
    if (head < tail) pending = int64_t(atomicAdd(&h->dq_head, 1u));
  }
  if (pending >= 0 && pending < int64_t(ws.L.qcap) &&
      ld_acquire_u32(&ws.ready()[pending])) {
    const QTask* e = ws.entries() + pending;
    t = QTask{__ldcg(&e->type), __ldcg(&e->b), __ldcg(&e->s), __ldcg(&e->aux)};
    pending = -1;
    return true;
  }
  const uint32_t total = uint32_t(ws.L.B) * uint32_t(ws.L.S);
  if (ld_volatile_u32(&h->p1_next) < total) {
    const uint32_t k = atomicAdd(&h->p1_next, 1u);
    if (k < total) {
      t = QTask{first_type, int(k / ws.L.S), int(k % ws.L.S), 0};
      return true;
    }
  }
  exhausted = true;
  return false;
}

// Producer back-off when no task is runnable. Returns false when production
// should stop: every row is done, the launch aborted, or nothing became
// runnable for kWaitNs (then the launch is aborted). `idle_t0` is the global
// time at which the current idle stretch began (0: not idle).
__device__ inline bool producer_idle(const Ws& ws, bool exhausted, uint64_t& idle_t0) {
  WsHeader* h = ws.hdr();
  if (ld_volatile_u32(&h->abort)) return false;
  if (exhausted && ld_volatile_u32(&h->rows_done) >= uint32_t(ws.L.B)) return false;
  const uint64_t now = global_ns();
  if (idle_t0 == 0) {
    idle_t0 = now;
  } else if (now - idle_t0 > kWaitNs) {
    atomicExch(&h->abort, 1u);
    return false;
  }
  __nanosleep(256);
  return true;
}

// ------------------------------------------------------------------ ring
// Per stage: which task (slot of the task table) and which piece of it.
struct ChunkMeta {
  int slot;    // task table slot; -1: end of stream
  int r;       // row index within the task
  int k;       // chunk index within the row slice
  int c0, c1;  // vector range [c0, c1) within the row
  int last_k;  // 1 when this is the last chunk of row r
  int last;    // 1 when this is the last chunk of the task
  int pad;
};

struct Ring {
  uint8_t* buf;         // kStages * kChunk bytes
  uint64_t* full;       // [kStages]
  uint64_t* empty;      // [kStages]
  ChunkMeta* meta;      // [kStages]
  QTask* ttab;          // [kStages] tasks in flight
  volatile int* abort;  // CTA-local abort flag
};

__device__ __forceinline__ void consumers_sync() { named_bar_sync(1, kCons); }

__device__ inline void ring_init(const Ring& r) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], kCW);
    }
    *r.abort = 0;
    fence_mbar_init();
  }
}

// Vector range of slice s of a row of nvec vectors cut into S slices.
__device__ __forceinline__ void slice_range(int nvec, int S, int s, int& v0, int& v1) {
  v0 = int(int64_t(nvec) * s / S);
  v1 = int(int64_t(nvec) * (s + 1) / S);
}

// Chunking of a row slice of nv vectors: chunks of cv vectors, cv a multiple of
// 32 (units of 32 vectors never straddle chunks) and cv * 16 <= kChunk.
__device__ __forceinline__ void chunking(int nv, int& nchunk, int& cv) {
  constexpr int kMaxCv = kChunk / 16;
  nchunk = nv > 0 ? (nv + kMaxCv - 1) / kMaxCv : 0;
  cv = nchunk > 0 ? ((nv + nchunk - 1) / nchunk + 31) / 32 * 32 : 0;
  if (cv > kMaxCv) cv = kMaxCv;
  if (nchunk > 0) nchunk = (nv + cv - 1) / cv;
}

// Producer: waits for stage `it` to be free, then fills its metadata.
__device__ __forceinline__ bool claim_stage(const Ring& ring, uint32_t it) {
  const int stage = it % kStages;
  if (it >= kStages && !mbar_wait(&ring.empty[stage], ((it / kStages) - 1) & 1)) {
    *ring.abort = 1;
    return false;
  }
  return true;
}

// Producer: streams the rows of one task (rows[] are row base pointers,
// `paired` interleaves chunk k of every row: r0k0, r1k0, r0k1, r1k1, ...).
__device__ inline bool produce_task(const Ring& ring, uint32_t& it, uint32_t& nt, const QTask& t,
                                    const char* const* rows, int nrows, bool paired, int v0,
                                    int v1) {
  // The table entry of task nt is reused by task nt + kStages; it is written
  // only once the task's first stage is claimed, i.e. after every consumer
  // warp released the stage kStages earlier and so has read the entry of every
  // task that started there or before (every task spans at least one stage).
  const int slot = int(nt % kStages);
  ++nt;
  int nchunk, cv;
  chunking(v1 - v0, nchunk, cv);
  const int total = nrows * nchunk;
  for (int q = 0; q < total; ++q, ++it) {
    const int r = paired ? (q % nrows) : (q / nchunk);
    const int k = paired ? (q / nrows) : (q % nchunk);
    if (!claim_stage(ring, it)) return false;
    if (q == 0) ring.ttab[slot] = t;
    const int stage = it % kStages;
    const int c0 = v0 + k * cv;
    const int c1 = min(v1, c0 + cv);
    ChunkMeta m;
    m.slot = slot;
    m.r = r;
    m.k = k;
    m.c0 = c0;
    m.c1 = c1;
    m.last_k = (k == nchunk - 1);
    m.last = (q == total - 1);
    m.pad = 0;
    ring.meta[stage] = m;
    const uint32_t bytes = uint32_t(c1 - c0) * 16u;
    mbar_arrive_expect_tx(&ring.full[stage], bytes);
    bulk_g2s(ring.buf + size_t(stage) * kChunk, rows[r] + size_t(c0) * 16, bytes,
             &ring.full[stage]);
  }
  return true;
}

// Producer: end-of-stream marker (a stage without data).
__device__ inline void produce_end(const Ring& ring, uint32_t& it) {
  if (!claim_stage(ring, it)) return;
  const int stage = it % kStages;
  ring.meta[stage].slot = -1;
  mbar_arrive(&ring.full[stage]);
  ++it;
}

// Consumers: wait for stage `it`; false on timeout.
__device__ __forceinline__ bool wait_stage(const Ring& ring, uint32_t it) {
  const int stage = it % kStages;
  if (*ring.abort || !mbar_wait(&ring.full[stage], (it / kStages) & 1)) {
    *ring.abort = 1;
    return false;
  }
  return true;
}

__device__ __forceinline__ void release_stage(const Ring& ring, uint32_t it) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&ring.empty[it % kStages]);
}

__device__ __forceinline__ const uint4* stage_data(const Ring& ring, uint32_t it) {
  return reinterpret_cast<const uint4*>(ring.buf + size_t(it % kStages) * kChunk);
}

}  // namespace sv
