// Sampling-mode verification kernel (spec_verify_sample).
//
// Method ("aiengineeringfromscratch.com - Speculative decoding and EAGLE-3",
// "Variant: Leviathan rejection sampling" and Steps 1-3): draft token d_i is
// accepted iff p_i(d_i) <= 0 or u_i < min(1, q_i(d_i)/p_i(d_i)); at the first
// rejection j the correction is drawn from (q_j - p_j)+ (q_j if that mass is
// zero); after K acceptances a bonus token is drawn from q_K. The draw is the
// inverse CDF in token-index order with the single uniform u_K.
//
// GB300 mapping. Persistent thread-block clusters; cluster c verifies batch
// rows c, c + ncl, ... The C CTAs of a cluster split the vocabulary into C
// contiguous slices. Per row:
//   1. pass 1: each CTA consumes its slice of the 2K logit rows (target and
//      draft, positions 0..K-1) from the bulk-copy ring (stream.cuh), keeping
//      per-thread running (max, sum of exp2); the producer thread is already
//      streaming the next row behind it;
//   2. per-CTA partials are all-gathered over distributed shared memory, so
//      every CTA holds the softmax statistics of all 2K rows and evaluates the
//      K accept tests; a warp ballot gives the first rejection j;
//   3. the final draw re-reads only row j of both tensors (hot in L2), or
//      target row K for a bonus (its statistics first): each CTA sums its
//      slice, keeping the sum of every 16-byte vector in shared memory; the
//      CTA sums are all-gathered and the CTA holding u_K * total mass finds
//      the token by a block scan over its vector sums;
//   4. CTA 0 writes the row's outputs.
// No global scratch memory is used.
//
// Arithmetic. No fp64 arithmetic (GB300 runs fp64 at a small fraction of its
// fp32 rate): logits are widened to fp32, exponentials use the MUFU exp2 with
// an integer offset ceil(max * log2(e)/T), and every sum a decision depends on
// is a float pair (df.cuh). A decision (an accept test, or the boundary of the
// drawn token) is taken from the fp32 path only when the uniform is farther
// from the threshold than twice a proven bound on that path's error;
// otherwise the row is recomputed with double-float exponentials (relative
// error < 4e-12 per term) and flagged in row_info. The result equals an
// exact-arithmetic evaluation except for rows flagged SPEC_ROW_UNCERTIFIED.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "../../include/specverify.h"
#include "cluster_launch.cuh"
#include "common.cuh"
#include "df.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "stream.cuh"

namespace sv {
namespace {

constexpr int kVsCap = 2048;  // vector sums kept per CTA (slice <= kVsCap vectors)
constexpr int kUnroll = 4;    // vectors in flight per thread in the direct-load sweeps

// ------------------------------------------------------------------ layout
struct Misc {
  int tok[kMaxK];
  float zt_d[kMaxK];  // target logit of the draft token, per position
  float zd_d[kMaxK];  // draft logit of the draft token
  float u[kMaxK + 1];
  int bad_token;
  int abort;
  int acc_state[kMaxK];
  float qd[kMaxK], pd[kMaxK];
  float src[16];  // this CTA's small exchange payload
  df wR[kCW];
  float wQ[kCW], wP[kCW], wAq[kCW], wAp[kCW];
  df scan[kCW];
  // scalars computed by one thread, read by all consumers
  int go;      // a sample point exists
  int cs;      // CTA holding the sample point
  df base;     // mass before CTA cs
  df tstar;    // u_K * total mass
  float E;     // error bound of the draw
  int zero_res;
  int token, cert, found;
};

struct Layout {
  Ring ring;
  Xc xc;
  Misc* misc;
  float* wM;  // [R][kCW]
  df* wS;     // [R][kCW]
  int* wBad;  // [R][kCW]
  float* rowM;
  float* rowKc;
  df* rowS;
  df* rowInv;
  int* rowOK;
  df* vsd;  // [kVsCap]
  float* tab_hi;
  float* tab_lo;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline int xc_floats(int R) { return 4 * R > 16 ? 4 * R : 16; }

template <class F>
__host__ __device__ inline size_t carve(int R, F&& put) {
  size_t o = size_t(kStages) * kChunk;  // ring at offset 0
  auto take = [&](size_t bytes, size_t al) {
    o = align_up(o, al);
    const size_t at = o;
    o += bytes;
    return at;
  };
  put(0, take((2 * kStages + 2) * 8, 8));                          // ring + exchange barriers
  put(1, take(sizeof(Misc), 16));                                  // misc
  put(2, take(size_t(R) * kCW * sizeof(df), 8));                   // wS
  put(3, take(size_t(R) * sizeof(df) * 2, 8));                     // rowS, rowInv
  put(4, take(size_t(kVsCap) * sizeof(df), 16));                   // vector sums
  put(5, take(size_t(2) * kMaxCluster * xc_floats(R) * 4, 16));    // exchange slots
  put(6, take(size_t(R) * kCW * 4 * 2, 4));                        // wM, wBad
  put(7, take(size_t(R) * 4 * 3, 4));                              // rowM, rowKc, rowOK
  put(8, take(256 * 4 * 2, 4));                                    // exp2 table
  return align_up(o, 128);
}

__host__ __device__ inline size_t sample_smem_bytes(int R) { return carve(R, [](int, size_t) {}); }

__device__ inline Layout make_layout(uint8_t* base, int R) {
  Layout L;
  L.ring.buf = base;
  L.xc.slot = xc_floats(R);
  carve(R, [&](int id, size_t at) {
    uint8_t* p = base + at;
    switch (id) {
      case 0:
        L.ring.full = reinterpret_cast<uint64_t*>(p);
        L.ring.empty = L.ring.full + kStages;
        L.xc.bar = L.ring.empty + kStages;
        break;
      case 1:
        L.misc = reinterpret_cast<Misc*>(p);
        L.ring.abort = &L.misc->abort;
        break;
      case 2:
        L.wS = reinterpret_cast<df*>(p);
        break;
      case 3:
        L.rowS = reinterpret_cast<df*>(p);
        L.rowInv = L.rowS + R;
        break;
      case 4:
        L.vsd = reinterpret_cast<df*>(p);
        break;
      case 5:
        L.xc.buf = reinterpret_cast<float*>(p);
        break;
      case 6:
        L.wM = reinterpret_cast<float*>(p);
        L.wBad = reinterpret_cast<int*>(L.wM + R * kCW);
        break;
      case 7:
        L.rowM = reinterpret_cast<float*>(p);
        L.rowKc = L.rowM + R;
        L.rowOK = reinterpret_cast<int*>(L.rowKc + R);
        break;
      case 8:
        L.tab_hi = reinterpret_cast<float*>(p);
        L.tab_lo = L.tab_hi + 256;
        break;
    }
  });
  return L;
}

// ------------------------------------------------------------------ arguments
struct Bounds {
  float ex2;     // relative error bound of ex2.approx.ftz.f32 on [-126, 1]
  float gamma1;  // relative error bound of the pass-1 fp32 summation
  float xbar;    // bound on sum_v q_v |x_v| before the row is swept (log2 V + 2)
};

struct SampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  int B, K, V;
  float c;         // fl32(log2(e) / T)
  float Chi, Clo;  // log2(e) / T as a float pair
  Bounds bd;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  int32_t* row_info;
  float* q_at_d;
  float* p_at_d;
};

enum { kAccept = 0, kReject = 1, kAmbiguous = 2, kInvalid = 3 };

// ------------------------------------------------------------------ pass-1 statistics
// Per-thread running max M, integer offset Kc = ceil(M c) and S = sum exp2(z c - Kc).
template <class E>
struct StatOp {
  float c;
  float M, Kc, S;
  int bad;
  int row_base;
  const Layout* L;
  __device__ void begin_row(int) {
    M = -INFINITY;
    Kc = -INFINITY;
    S = 0.0f;
    bad = 0;
  }
  __device__ __forceinline__ void vec(const uint4& v, int) {
    const float vm = E::vmax(v);
    if (vm != vm) {
      bad = 1;
      return;
    }
    if (vm > M) {
      const float Kn = offset_of(vm, c);
      if (S != 0.0f) S = __fmul_rn(S, pow2i(__fsub_rn(Kc, Kn)));
      M = vm;
      Kc = Kn;
    }
    if (Kc == -INFINITY) return;  // only -inf logits so far
    float z[E::kVec];
    E::unpack(v, z);
    float e[E::kVec];
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) e[k] = ex2_approx(__fmaf_rn(z[k], c, -Kc));
#pragma unroll
    for (int w = 1; w < E::kVec; w <<= 1)
#pragma unroll
      for (int k = 0; k < E::kVec; k += 2 * w) e[k] = __fadd_rn(e[k], e[k + w]);
    S = __fadd_rn(S, e[0]);
  }
  __device__ void end_row(int r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float Mw = warp_max_f(M);
    df s{0.f, 0.f};
    if (S != 0.0f) s.hi = __fmul_rn(S, pow2i(__fsub_rn(Kc, offset_of(Mw, c))));
    s = df_warp_sum(s);
    const int anybad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      const int rr = row_base + r;
      L->wM[rr * kCW + warp] = Mw;
      L->wS[rr * kCW + warp] = s;
      L->wBad[rr * kCW + warp] = anybad;
    }
  }
};

// Consumers: the CTA partial (M, S.hi, S.lo, bad) of rows [r0, r1) into the
// exchange payload at float offset 4*(r - r0).
__device__ void stats_payload(const Layout& L, int r0, int r1, float c, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = r0 + warp; r < r1; r += kCW) {
    const float m = lane < kCW ? L.wM[r * kCW + lane] : -INFINITY;
    df s = lane < kCW ? L.wS[r * kCW + lane] : df{0.f, 0.f};
    const int bw = lane < kCW ? L.wBad[r * kCW + lane] : 0;
    const float Mc = warp_max_f(m);
    if (s.hi != 0.0f) {
      const float sc = pow2i(__fsub_rn(offset_of(m, c), offset_of(Mc, c)));
      s = {__fmul_rn(s.hi, sc), __fmul_rn(s.lo, sc)};
    }
    s = df_warp_sum(s);
    const int bad = __any_sync(0xffffffffu, bw);
    if (lane == 0) {
      float* o = out + 4 * (r - r0);
      o[0] = Mc;
      o[1] = s.hi;
      o[2] = s.lo;
      o[3] = __int_as_float(bad);
    }
  }
}

// Final statistics of rows [r0, r1) from the gathered payloads of exchange e
// (same values, same order in every CTA: bit-identical results everywhere).
__device__ void stats_final(const Layout& L, uint32_t e, int r0, int r1, float c, int csize) {
  for (int r = r0 + int(threadIdx.x); r < r1; r += kCons) {
    const int o = 4 * (r - r0);
    float M = -INFINITY;
    int bad = 0;
    for (int q = 0; q < csize; ++q) {
      const float* s = xc_slot(L.xc, e, q) + o;
      M = fmaxf(M, s[0]);
      bad |= __float_as_int(s[3]);
    }
    const float Kc = offset_of(M, c);
    df S{0.f, 0.f};
    for (int q = 0; q < csize; ++q) {
      const float* s = xc_slot(L.xc, e, q) + o;
      if (s[1] != 0.0f) {
        const float sc = pow2i(__fsub_rn(offset_of(s[0], c), Kc));
        S = df_add(S, df{__fmul_rn(s[1], sc), __fmul_rn(s[2], sc)});
      }
    }
    const bool ok = !bad && isfinite(M) && fabsf(Kc) < 4194304.0f && S.hi > 0.0f && isfinite(S.hi);
    L.rowM[r] = M;
    L.rowKc[r] = Kc;
    L.rowS[r] = S;
    L.rowInv[r] = ok ? df_recip(S) : df{0.f, 0.f};
    L.rowOK[r] = ok ? 1 : 0;
  }
}

// Full statistics exchange of rows [r0, r1): payload, all-gather, final.
__device__ bool stats_exchange(const Layout& L, uint32_t& e, int r0, int r1, float c, int crank,
                               int csize, float* scratch) {
  stats_payload(L, r0, r1, c, scratch);
  consumers_sync();
  if (threadIdx.x < 32) xc_push(L.xc, e, scratch, 4 * (r1 - r0), crank, csize);
  const bool ok = xc_wait(L.xc, e, L.ring.abort);
  if (ok) stats_final(L, e, r0, r1, c, csize);
  ++e;
  consumers_sync();
  return ok;
}

// Statistics of one row slice read directly from global memory (bonus row).
template <class E>
__device__ void stats_direct(const typename E::T* row, int vbeg, int vend, StatOp<E>& op) {
  const uint4* p = reinterpret_cast<const uint4*>(row);
  op.begin_row(0);
  for (int v0 = vbeg + int(threadIdx.x); v0 < vend; v0 += kCons * kUnroll) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (v0 + u * kCons < vend) buf[u] = ldg_nc_v4(p + v0 + u * kCons);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (v0 + u * kCons < vend) op.vec(buf[u], v0 + u * kCons);
  }
  op.end_row(0);
}

// ------------------------------------------------------------------ accurate path
// 2^(z C - Kc) in pair arithmetic (C = log2(e)/T as Chi + Clo, Kc an integer).
__device__ __forceinline__ df acc_elem(float z, float Chi, float Clo, float Kc, const float* th,
                                       const float* tl) {
  const df p = two_prod(z, Chi);
  const float pl = __fmaf_rn(z, Clo, p.lo);
  const df s = two_sum(p.hi, -Kc);
  return df_exp2(s.hi, __fadd_rn(s.lo, pl), th, tl);
}

// Relative error bound of one normalised double-float term q_v or p_v: the
// exponential (< 4e-13), its argument (< 2^-46 (|z C| + |Kc|) < 1e-12 for
// offsets below 2^22, the row check), the normaliser sum and reciprocal
// (< 1e-12); kept above their total.
constexpr float kAccRho = 4e-12f;

__device__ inline void load_table(const Layout& L) {
  for (int i = threadIdx.x; i < 256; i += kCons) {
    L.tab_hi[i] = kExp2Tab.hi[i];
    L.tab_lo[i] = kExp2Tab.lo[i];
  }
}

// Accurate sum_v 2^(z_v C - Kc) over the whole row for up to two rows (row1
// may be null). Consumers only; every CTA returns the same pairs.
template <class E>
__device__ bool acc_norms(const Layout& L, uint32_t& e, const typename E::T* row0, float Kc0,
                          const typename E::T* row1, float Kc1, int vbeg, int vend,
                          const SampleArgs& a, int crank, int csize, df* out) {
  Misc& ms = *L.misc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  df a0{0.f, 0.f}, a1{0.f, 0.f};
  const uint4* p0 = reinterpret_cast<const uint4*>(row0);
  const uint4* p1 = reinterpret_cast<const uint4*>(row1);
  for (int vi = vbeg + tid; vi < vend; vi += kCons) {
    float z[E::kVec];
    E::unpack(ldg_nc_v4(p0 + vi), z);
#pragma unroll
    for (int k = 0; k < E::kVec; ++k)
      a0 = df_add(a0, acc_elem(z[k], a.Chi, a.Clo, Kc0, L.tab_hi, L.tab_lo));
    if (row1) {
      E::unpack(ldg_nc_v4(p1 + vi), z);
#pragma unroll
      for (int k = 0; k < E::kVec; ++k)
        a1 = df_add(a1, acc_elem(z[k], a.Chi, a.Clo, Kc1, L.tab_hi, L.tab_lo));
    }
  }
  a0 = df_warp_sum(a0);
  a1 = df_warp_sum(a1);
  if (lane == 0) {
    ms.scan[warp] = a0;
    ms.wR[warp] = a1;
  }
  consumers_sync();
  if (tid == 0) {
    df s0{0.f, 0.f}, s1{0.f, 0.f};
    for (int w = 0; w < kCW; ++w) {
      s0 = df_add(s0, ms.scan[w]);
      s1 = df_add(s1, ms.wR[w]);
    }
    ms.src[0] = s0.hi;
    ms.src[1] = s0.lo;
    ms.src[2] = s1.hi;
    ms.src[3] = s1.lo;
  }
  consumers_sync();
  if (tid < 32) xc_push(L.xc, e, ms.src, 4, crank, csize);
  const bool ok = xc_wait(L.xc, e, L.ring.abort);
  df t0{0.f, 0.f}, t1{0.f, 0.f};
  for (int q = 0; q < csize; ++q) {
    const float* s = xc_slot(L.xc, e, q);
    t0 = df_add(t0, df{s[0], s[1]});
    t1 = df_add(t1, df{s[2], s[3]});
  }
  out[0] = t0;
  out[1] = t1;
  ++e;
  consumers_sync();
  return ok;
}

// ------------------------------------------------------------------ final draw entries
// fp32 path: r = max(0, q - p) with q = exp2(z c - Kc_q) / S_q (or r = q).
template <class E>
struct FastEntries {
  const uint4* tq;
  const uint4* tp;  // null: draw from q
  float c, Kq, Rq, Kp, Rp;
  // r[k] from loaded vectors; returns their pairwise fp32 sum and accumulates
  // sum q, sum p, sum q|x|, sum p|x|.
  __device__ __forceinline__ float run(const uint4& vq, const uint4& vp, float (&r)[E::kVec],
                                       float& qs, float& ps, float& aq, float& ap) const {
    float zq[E::kVec], zp[E::kVec];
    E::unpack(vq, zq);
    if (tp) E::unpack(vp, zp);
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      const float xa = __fmaf_rn(zq[k], c, -Kq);
      const float q = __fmul_rn(ex2_approx(xa), Rq);
      qs = __fadd_rn(qs, q);
      aq = __fmaf_rn(q, fminf(fabsf(xa), 1.0e4f), aq);
      if (tp) {
        const float xb = __fmaf_rn(zp[k], c, -Kp);
        const float p = __fmul_rn(ex2_approx(xb), Rp);
        ps = __fadd_rn(ps, p);
        ap = __fmaf_rn(p, fminf(fabsf(xb), 1.0e4f), ap);
        r[k] = fmaxf(__fsub_rn(q, p), 0.0f);
      } else {
        r[k] = q;
      }
    }
    float t[E::kVec];
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) t[k] = r[k];
#pragma unroll
    for (int w = 1; w < E::kVec; w <<= 1)
#pragma unroll
      for (int k = 0; k < E::kVec; k += 2 * w) t[k] = __fadd_rn(t[k], t[k + w]);
    return t[0];
  }
  // entries of vector vi as pairs, and the vector sum the sweep recorded
  __device__ __forceinline__ df entries(int vi, df (&rd)[E::kVec]) const {
    float r[E::kVec];
    float a = 0.f, b = 0.f, cc = 0.f, d = 0.f;
    const uint4 vq = ldg_nc_v4(tq + vi);
    const uint4 vp = tp ? ldg_nc_v4(tp + vi) : vq;
    const float vs = run(vq, vp, r, a, b, cc, d);
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) rd[k] = {r[k], 0.f};
    return {vs, 0.f};
  }
};

// double-float path.
template <class E>
struct AccEntries {
  const uint4* tq;
  const uint4* tp;
  float Chi, Clo, Kq, Kp;
  df Iq, Ip;  // accurate 1/S of the two rows
  const float* th;
  const float* tl;
  __device__ __forceinline__ df run(const uint4& vq, const uint4& vp, df (&r)[E::kVec], float& qs,
                                    float& ps) const {
    float zq[E::kVec], zp[E::kVec];
    E::unpack(vq, zq);
    if (tp) E::unpack(vp, zp);
    df vs{0.f, 0.f};
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      const df q = df_mul(acc_elem(zq[k], Chi, Clo, Kq, th, tl), Iq);
      qs = __fadd_rn(qs, q.hi);
      df rk = q;
      if (tp) {
        const df p = df_mul(acc_elem(zp[k], Chi, Clo, Kp, th, tl), Ip);
        ps = __fadd_rn(ps, p.hi);
        rk = df_sub(q, p);
        if (!(rk.hi > 0.0f)) rk = {0.f, 0.f};
      }
      r[k] = rk;
      vs = df_add(vs, rk);
    }
    return vs;
  }
  __device__ __forceinline__ df entries(int vi, df (&rd)[E::kVec]) const {
    float a = 0.f, b = 0.f;
    const uint4 vq = ldg_nc_v4(tq + vi);
    const uint4 vp = tp ? ldg_nc_v4(tp + vi) : vq;
    return run(vq, vp, rd, a, b);
  }
};

// ------------------------------------------------------------------ draw search
// Block-wide exclusive scan of one pair per consumer thread (in thread order).
__device__ df block_excl_scan_df(Misc& ms, df v, df& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  df inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const df y = df_shfl_up(inc, o);
    if (lane >= o) inc = df_add(inc, y);
  }
  if (lane == 31) ms.scan[warp] = inc;
  consumers_sync();
  df pre{0.f, 0.f};
  total = {0.f, 0.f};
  for (int w = 0; w < kCW; ++w) {
    if (w == warp) pre = total;
    total = df_add(total, ms.scan[w]);
  }
  consumers_sync();
  return df_add(pre, df_sub(inc, v));
}

// CTA ms.cs: find the entry holding t = ms.tstar, using the per-vector sums in
// L.vsd (nv <= kVsCap) and recomputing only the vector that holds it. Thread
// 0..kCons-1 call; the result lands in ms.token / ms.cert (certified iff both
// boundaries are farther than 2E from t).
template <int kVec, class Entries>
__device__ void block_search(const Layout& L, int vbeg, int vend, const Entries& ent) {
  Misc& ms = *L.misc;
  const int tid = threadIdx.x;
  const int nv = vend - vbeg;
  const int seg = (nv + kCons - 1) / kCons;
  const int s0 = min(nv, tid * seg), s1 = min(nv, s0 + seg);
  df s{0.f, 0.f};
  for (int i = s0; i < s1; ++i) s = df_add(s, L.vsd[i]);
  df total;
  const df excl = block_excl_scan_df(ms, s, total);
  const df lo = df_add(ms.base, excl);
  const df hi = df_add(lo, s);
  const df t = ms.tstar;
  // first thread whose segment ends past t; else the last thread with mass
  if (tid == 0) ms.found = INT_MAX;
  consumers_sync();
  if (s.hi > 0.0f && df_gt(hi, t)) atomicMin(&ms.found, tid);
  consumers_sync();
  if (ms.found == INT_MAX) {
    if (tid == 0) ms.found = -1;
    consumers_sync();
    if (s.hi > 0.0f) atomicMax(&ms.found, tid);
    consumers_sync();
  }
  if (tid == ms.found) {
    // walk this segment's vectors, then the entries of the vector holding t
    df cum = lo;
    int vsel = -1, vlast = -1;
    df vlo = lo, vlast_lo = lo;
    for (int i = s0; i < s1; ++i) {
      const df nx = df_add(cum, L.vsd[i]);
      if (L.vsd[i].hi > 0.0f) {
        vlast = i;
        vlast_lo = cum;
        if (df_gt(nx, t)) {
          vsel = i;
          vlo = cum;
          break;
        }
      }
      cum = nx;
    }
    if (vsel < 0) {
      vsel = vlast;
      vlo = vlast_lo;
    }
    int token = -1;
    df tlo = vlo, thi = vlo;
    if (vsel >= 0) {
      df r[kVec];
      ent.entries(vbeg + vsel, r);
      df c0 = vlo;
      int lastk = -1;
      df llo = vlo, lhi = vlo;
      for (int k = 0; k < kVec; ++k) {
        const df c1 = df_add(c0, r[k]);
        if (r[k].hi > 0.0f) {
          lastk = k;
          llo = c0;
          lhi = c1;
          if (token < 0 && df_gt(c1, t)) {
            token = (vbeg + vsel) * kVec + k;
            tlo = c0;
            thi = c1;
          }
        }
        c0 = c1;
      }
      if (token < 0 && lastk >= 0) {
        token = (vbeg + vsel) * kVec + lastk;
        tlo = llo;
        thi = lhi;
      }
    }
    const float m1 = df_sub(t, tlo).hi, m2 = df_sub(thi, t).hi;
    ms.token = token;
    ms.cert = (token >= 0 && fminf(m1, m2) > 2.02f * ms.E) ? 1 : 0;
  }
  consumers_sync();
}

// CTA ms.cs when its slice exceeds the vector-sum buffer: warp 0 walks the
// whole slice (lanes on consecutive vectors) for the entry holding t.
template <int kVec, class Entries>
__device__ void warp_walk_search(const Layout& L, int vbeg, int vend, const Entries& ent) {
  Misc& ms = *L.misc;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const df t = ms.tstar;
    df base = ms.base;
    int tokn = -1, lastk = -1;
    df tlo = base, thi = base, llo = base, lhi = base;
    for (int v0 = vbeg; v0 < vend && tokn < 0; v0 += 32) {
      const int vi = v0 + lane;
      df r[kVec];
      df vs{0.f, 0.f};
      if (vi < vend) {
        vs = ent.entries(vi, r);
      } else {
#pragma unroll
        for (int k = 0; k < kVec; ++k) r[k] = {0.f, 0.f};
      }
      df inc = vs;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const df y = df_shfl_up(inc, o);
        if (lane >= o) inc = df_add(inc, y);
      }
      df c0 = df_add(base, df_sub(inc, vs));
      int tk = -1, lk = -1;
      df lo{0.f, 0.f}, hi{0.f, 0.f}, l0{0.f, 0.f}, l1{0.f, 0.f};
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const df c1 = df_add(c0, r[k]);
        if (r[k].hi > 0.0f) {
          lk = vi * kVec + k;
          l0 = c0;
          l1 = c1;
          if (tk < 0 && df_gt(c1, t)) {
            tk = vi * kVec + k;
            lo = c0;
            hi = c1;
          }
        }
        c0 = c1;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, tk >= 0);
      if (hit) {
        const int l = __ffs(int(hit)) - 1;
        tokn = __shfl_sync(0xffffffffu, tk, l);
        tlo = df_shfl(lo, l);
        thi = df_shfl(hi, l);
      }
      const unsigned has = __ballot_sync(0xffffffffu, lk >= 0);
      if (has) {
        const int l = 31 - __clz(int(has));
        lastk = __shfl_sync(0xffffffffu, lk, l);
        llo = df_shfl(l0, l);
        lhi = df_shfl(l1, l);
      }
      base = df_add(base, df_shfl(inc, 31));
    }
    if (tokn < 0) {
      tokn = lastk;
      tlo = llo;
      thi = lhi;
    }
    if (lane == 0) {
      const float m1 = df_sub(t, tlo).hi, m2 = df_sub(thi, t).hi;
      ms.token = tokn;
      ms.cert = (tokn >= 0 && fminf(m1, m2) > 2.02f * ms.E) ? 1 : 0;
    }
  }
  consumers_sync();
}

// Thread 0: locate the CTA holding t among the gathered CTA sums of exchange e
// (floats 0, 1 of each slot).
__device__ void locate_cta(const Layout& L, uint32_t e, int csize) {
  Misc& ms = *L.misc;
  int cs = -1;
  df pre{0.f, 0.f}, pre_cs{0.f, 0.f};
  for (int q = 0; q < csize; ++q) {
    const float* s = xc_slot(L.xc, e, q);
    const df x{s[0], s[1]};
    const df nx = df_add(pre, x);
    if (x.hi > 0.0f) {
      cs = q;
      pre_cs = pre;
      if (df_gt(nx, ms.tstar)) break;
    }
    pre = nx;
  }
  ms.cs = cs;
  ms.base = pre_cs;
}

// After a search: every CTA learns the token and its certification.
__device__ bool publish_draw(const Layout& L, uint32_t& e, int crank, int csize, int& token,
                             int& cert) {
  Misc& ms = *L.misc;
  if (threadIdx.x == 0) {
    const bool mine = ms.go && ms.cs == crank;
    ms.src[0] = __int_as_float(mine ? ms.token : -2);
    ms.src[1] = __int_as_float(mine ? ms.cert : 0);
  }
  consumers_sync();
  if (threadIdx.x < 32) xc_push(L.xc, e, ms.src, 2, crank, csize);
  const bool ok = xc_wait(L.xc, e, L.ring.abort);
  token = -1;
  cert = 0;
  for (int q = 0; q < csize; ++q) {
    const float* s = xc_slot(L.xc, e, q);
    if (__float_as_int(s[0]) != -2) {
      token = __float_as_int(s[0]);
      cert = __float_as_int(s[1]);
    }
  }
  ++e;
  consumers_sync();
  return ok;
}

// ------------------------------------------------------------------ one row
template <class E>
__device__ void verify_row(const SampleArgs& a, const Layout& L, int b, int vbeg, int vend,
                           int crank, int csize, uint32_t& it, uint32_t& e) {
  using T = typename E::T;
  Misc& ms = *L.misc;
  const int K = a.K, V = a.V;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const T* tgt = static_cast<const T*>(a.target) + size_t(b) * (K + 1) * V;
  const T* drf = static_cast<const T*>(a.draft) + size_t(b) * K * V;
  const float c = a.c;

  if (warp == 1) {
    int bad = 0;
    if (lane < K) {
      const int d = a.tokens[size_t(b) * K + lane];
      ms.tok[lane] = d;
      if (d < 0 || d >= V) {
        bad = 1;
        ms.zt_d[lane] = 0.f;
        ms.zd_d[lane] = 0.f;
      } else {
        ms.zt_d[lane] = E::load(tgt + size_t(lane) * V, d);
        ms.zd_d[lane] = E::load(drf + size_t(lane) * V, d);
      }
    }
    if (lane <= K) ms.u[lane] = a.uniforms[size_t(b) * (K + 1) + lane];
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) ms.bad_token = bad;
  }

  // ---------------------------------------------------------------- pass 1
  StatOp<E> op;
  op.c = c;
  op.row_base = 0;
  op.L = &L;
  it = consume_rows(L.ring, it, 2 * K, vbeg, vend, op);
  consumers_sync();
  float* scratch = reinterpret_cast<float*>(L.vsd);  // payload staging (vsd is free here)
  bool alive = stats_exchange(L, e, 0, 2 * K, c, crank, csize, scratch);

  // ---------------------------------------------------------------- accept tests
  if (warp == 0 && lane < K) {
    const int i = lane, rt = 2 * i, rd = 2 * i + 1;
    int st;
    float qd = -1.f, pd = -1.f;
    if (ms.bad_token || !L.rowOK[rt] || !L.rowOK[rd]) {
      st = kInvalid;
    } else {
      const float zt = ms.zt_d[i], zd = ms.zd_d[i], u = ms.u[i];
      const float xt = __fmaf_rn(zt, c, -L.rowKc[rt]);
      const float xd = __fmaf_rn(zd, c, -L.rowKc[rd]);
      qd = __fmul_rn(ex2_approx(xt), L.rowInv[rt].hi);
      pd = __fmul_rn(ex2_approx(xd), L.rowInv[rd].hi);
      if (zd == -INFINITY) {
        st = kAccept;  // p(d) = 0 accepts
      } else if (zt == -INFINITY) {
        st = kReject;  // q(d) = 0: u < 0 never holds
      } else if (u == 0.0f) {
        st = kAccept;  // 0 < q(d)/p(d) whenever q(d) > 0
      } else {
        // ratio = 2^(xt - xd) * S_d / S_t; relative error bound: exp2, the
        // arguments (with the fp32 temperature constant), both row sums, and
        // five roundings
        const float ar = __fsub_rn(xt, xd);
        const float ratio = __fmul_rn(__fmul_rn(ex2_approx(ar), L.rowS[rd].hi), L.rowInv[rt].hi);
        const float dS = a.bd.ex2 + kLn2f * kU * a.bd.xbar + a.bd.gamma1;
        const float beta =
            1.1f * (a.bd.ex2 + 6.0f * kU + 2.0f * dS +
                    kLn2f * kU * (2.0f * fabsf(xt) + 2.0f * fabsf(xd) + fabsf(ar) +
                                  2.0f * a.bd.xbar + 4.0f));
        if (!(ar < 126.0f) || ratio >= 1.0f / (1.0f - beta)) {
          st = kAccept;  // ratio >= 1 for certain
        } else {
          const float rlo = fminf(1.0f, __fmul_rn(ratio, 1.0f - beta));
          const float rhi = fminf(1.0f, __fmul_rn(ratio, 1.0f + beta));
          st = (u < rlo) ? kAccept : (u >= rhi && ar > -120.0f ? kReject : kAmbiguous);
        }
      }
    }
    ms.acc_state[i] = st;
    ms.qd[i] = qd;
    ms.pd[i] = pd;
  }
  consumers_sync();

  int flags = 0, n = 0;
  bool error = ms.bad_token != 0 || !alive;
  while (!error) {
    int i = n;
    while (i < K && ms.acc_state[i] == kAccept) ++i;
    if (i == K) {
      n = K;
      break;
    }
    const int st = ms.acc_state[i];
    n = i;
    if (st == kInvalid) {
      error = true;
      break;
    }
    if (st == kReject) break;
    // ambiguous: decide with accurate row sums of target and draft row i
    flags |= SPEC_ROW_ACCEPT_REFINED;
    load_table(L);
    consumers_sync();
    df S2[2];
    alive = acc_norms<E>(L, e, tgt + size_t(i) * V, L.rowKc[2 * i], drf + size_t(i) * V,
                         L.rowKc[2 * i + 1], vbeg, vend, a, crank, csize, S2);
    if (!alive) {
      error = true;
      break;
    }
    // ratio = 2^((zt C - Kt) - (zd C - Kd)) * S_d / S_t in pair arithmetic
    const float zt = ms.zt_d[i], zd = ms.zd_d[i], u = ms.u[i];
    const df xt = df_add_f(df_add(two_prod(zt, a.Chi), df{__fmul_rn(zt, a.Clo), 0.f}), -L.rowKc[2 * i]);
    const df xd =
        df_add_f(df_add(two_prod(zd, a.Chi), df{__fmul_rn(zd, a.Clo), 0.f}), -L.rowKc[2 * i + 1]);
    const df ar = df_sub(xt, xd);
    bool acc;
    if (ar.hi >= 127.0f) {
      acc = true;
    } else if (ar.hi < -126.0f) {
      acc = false;  // ratio < 2^-100 < u (u > 0 here)
    } else {
      const df ratio =
          df_mul(df_mul(df_exp2(ar.hi, ar.lo, L.tab_hi, L.tab_lo), S2[1]), df_recip(S2[0]));
      acc = (ratio.hi >= 1.0f) || df_gt(ratio, df{u, 0.f});
      if (fabsf(__fsub_rn(u, fminf(1.0f, ratio.hi))) <= 1e-10f * ratio.hi) flags |= SPEC_ROW_UNCERTIFIED;
    }
    if (!acc) break;
    if (tid == 0) ms.acc_state[i] = kAccept;
    consumers_sync();
    n = i + 1;
  }

  // ---------------------------------------------------------------- final draw
  int token = -1;
  if (!error) {
    const bool bonus = (n == K);
    const int rq = bonus ? 2 * K : 2 * n;
    const int rpd = bonus ? -1 : 2 * n + 1;
    if (bonus) {
      StatOp<E> opk;
      opk.c = c;
      opk.row_base = 2 * K;
      opk.L = &L;
      stats_direct<E>(tgt + size_t(K) * V, vbeg, vend, opk);
      consumers_sync();
      alive = stats_exchange(L, e, 2 * K, 2 * K + 1, c, crank, csize, scratch);
      if (!alive || !L.rowOK[2 * K]) error = true;
    }
    if (!error) {
      const int jrow = bonus ? K : n;
      const uint4* vq = reinterpret_cast<const uint4*>(tgt + size_t(jrow) * V);
      const uint4* vp = bonus ? nullptr : reinterpret_cast<const uint4*>(drf + size_t(n) * V);
      const float uK = ms.u[K];
      const int nv = vend - vbeg;
      const bool keep = nv <= kVsCap;

      // ---------------- fp32 sweep, per-vector sums kept for the search
      FastEntries<E> fe;
      fe.tq = vq;
      fe.tp = vp;
      fe.c = c;
      fe.Kq = L.rowKc[rq];
      fe.Rq = L.rowInv[rq].hi;
      fe.Kp = bonus ? 0.f : L.rowKc[rpd];
      fe.Rp = bonus ? 0.f : L.rowInv[rpd].hi;
      {
        df acc{0.f, 0.f};
        float Q = 0.f, P = 0.f, Aq = 0.f, Ap = 0.f;
        for (int v0 = vbeg + tid; v0 < vend; v0 += kCons * kUnroll) {
          uint4 bq[kUnroll], bp[kUnroll];
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int vi = v0 + u * kCons;
            if (vi < vend) {
              bq[u] = ldg_nc_v4(vq + vi);
              bp[u] = vp ? ldg_nc_v4(vp + vi) : bq[u];
            }
          }
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int vi = v0 + u * kCons;
            if (vi < vend) {
              float r[E::kVec];
              const float vs = fe.run(bq[u], bp[u], r, Q, P, Aq, Ap);
              if (keep) L.vsd[vi - vbeg] = {vs, 0.f};
              acc = df_add_f(acc, vs);
            }
          }
        }
        acc = df_warp_sum(acc);
        Q = warp_sum_f(Q);
        P = warp_sum_f(P);
        Aq = warp_sum_f(Aq);
        Ap = warp_sum_f(Ap);
        if (lane == 0) {
          ms.wR[warp] = acc;
          ms.wQ[warp] = Q;
          ms.wP[warp] = P;
          ms.wAq[warp] = Aq;
          ms.wAp[warp] = Ap;
        }
      }
      consumers_sync();
      if (tid == 0) {
        df Rc{0.f, 0.f};
        float Qc = 0.f, Pc = 0.f, Aqc = 0.f, Apc = 0.f;
        for (int w = 0; w < kCW; ++w) {
          Rc = df_add(Rc, ms.wR[w]);
          Qc += ms.wQ[w];
          Pc += ms.wP[w];
          Aqc += ms.wAq[w];
          Apc += ms.wAp[w];
        }
        ms.src[0] = Rc.hi;
        ms.src[1] = Rc.lo;
        ms.src[2] = Qc;
        ms.src[3] = Pc;
        ms.src[4] = Aqc;
        ms.src[5] = Apc;
      }
      consumers_sync();
      if (tid < 32) xc_push(L.xc, e, ms.src, 6, crank, csize);
      alive = xc_wait(L.xc, e, L.ring.abort);
      if (tid == 0) {
        df Sr{0.f, 0.f};
        float Qt = 0.f, Pt = 0.f, Aqt = 0.f, Apt = 0.f;
        for (int q = 0; q < csize; ++q) {
          const float* s = xc_slot(L.xc, e, q);
          Sr = df_add(Sr, df{s[0], s[1]});
          Qt += s[2];
          Pt += s[3];
          Aqt += s[4];
          Apt += s[5];
        }
        // Error bound (probability units) of the fp32 sweep. Per term,
        // relative: exp2 (ex2), argument rounding and the fp32 temperature
        // constant (ln2 u |x| each), 1/S and the product (3u), and the row sum
        // behind 1/S (ex2 + ln2 u sum q|x| + gamma1); weights q (resp. p).
        auto side = [&](float Qs, float A) {
          const float xb = A / fmaxf(Qs, 1e-30f) + 1.0f;
          return 1.05f * fmaxf(Qs, 1.0f) *
                 (2.0f * a.bd.ex2 + 3.0f * kU + a.bd.gamma1 + kLn2f * kU * 4.0f * xb);
        };
        const float E = side(Qt, Aqt) + (bonus ? 0.f : side(Pt, Apt)) + 5.0f * kU * Sr.hi + 1e-30f;
        ms.E = E;
        ms.tstar = df_mul_f(Sr, uK);
        ms.go = (alive && Sr.hi > 2.0f * E) ? 1 : 0;
        if (ms.go) locate_cta(L, e, csize);
      }
      ++e;
      consumers_sync();
      if (ms.go && ms.cs == crank) {
        if (keep) block_search<E::kVec>(L, vbeg, vend, fe);
        else warp_walk_search<E::kVec>(L, vbeg, vend, fe);
      }
      consumers_sync();
      int cert = 0;
      alive = publish_draw(L, e, crank, csize, token, cert) && alive;
      if (!alive) error = true;

      if (!error && !cert) {
        // ---------------- double-float path
        flags |= SPEC_ROW_SAMPLE_REFINED;
        load_table(L);
        consumers_sync();
        df S2[2];
        alive = acc_norms<E>(L, e, tgt + size_t(jrow) * V, L.rowKc[rq],
                             bonus ? nullptr : drf + size_t(n) * V, bonus ? 0.f : L.rowKc[rpd],
                             vbeg, vend, a, crank, csize, S2);
        AccEntries<E> ae;
        ae.tq = vq;
        ae.tp = vp;
        ae.Chi = a.Chi;
        ae.Clo = a.Clo;
        ae.Kq = L.rowKc[rq];
        ae.Kp = bonus ? 0.f : L.rowKc[rpd];
        ae.Iq = df_recip(S2[0]);
        ae.Ip = bonus ? df{0.f, 0.f} : df_recip(S2[1]);
        ae.th = L.tab_hi;
        ae.tl = L.tab_lo;
        for (int pass = 0; pass < 2 && alive; ++pass) {
          df acc{0.f, 0.f};
          float Q = 0.f, P = 0.f;
          for (int v0 = vbeg + tid; v0 < vend; v0 += kCons * kUnroll) {
            uint4 bq[kUnroll], bp[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
              const int vi = v0 + u * kCons;
              if (vi < vend) {
                bq[u] = ldg_nc_v4(vq + vi);
                bp[u] = ae.tp ? ldg_nc_v4(vp + vi) : bq[u];
              }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
              const int vi = v0 + u * kCons;
              if (vi < vend) {
                df r[E::kVec];
                const df vs = ae.run(bq[u], bp[u], r, Q, P);
                if (keep) L.vsd[vi - vbeg] = vs;
                acc = df_add(acc, vs);
              }
            }
          }
          acc = df_warp_sum(acc);
          Q = warp_sum_f(Q);
          P = warp_sum_f(P);
          if (lane == 0) {
            ms.wR[warp] = acc;
            ms.wQ[warp] = Q;
            ms.wP[warp] = P;
          }
          consumers_sync();
          if (tid == 0) {
            df Rc{0.f, 0.f};
            float Qc = 0.f, Pc = 0.f;
            for (int w = 0; w < kCW; ++w) {
              Rc = df_add(Rc, ms.wR[w]);
              Qc += ms.wQ[w];
              Pc += ms.wP[w];
            }
            ms.src[0] = Rc.hi;
            ms.src[1] = Rc.lo;
            ms.src[2] = Qc;
            ms.src[3] = Pc;
          }
          consumers_sync();
          if (tid < 32) xc_push(L.xc, e, ms.src, 4, crank, csize);
          alive = xc_wait(L.xc, e, L.ring.abort);
          if (tid == 0) {
            df Sr{0.f, 0.f};
            float Qt = 0.f, Pt = 0.f;
            for (int q = 0; q < csize; ++q) {
              const float* s = xc_slot(L.xc, e, q);
              Sr = df_add(Sr, df{s[0], s[1]});
              Qt += s[2];
              Pt += s[3];
            }
            ms.zero_res = (Sr.hi == 0.0f && ae.tp != nullptr) ? 1 : 0;
            ms.E = kAccRho * (Qt + Pt) + 1e-14f * Sr.hi + 1e-36f;
            ms.tstar = df_mul_f(Sr, uK);
            ms.go = (alive && Sr.hi > 0.0f) ? 1 : 0;
            if (ms.go) locate_cta(L, e, csize);
          }
          ++e;
          consumers_sync();
          if (ms.zero_res) {
            // zero residual mass: the draw uses q_j itself
            flags |= SPEC_ROW_ZERO_RESIDUAL;
            ae.tp = nullptr;
            continue;
          }
          if (ms.go && ms.cs == crank) {
            if (keep) block_search<E::kVec>(L, vbeg, vend, ae);
            else warp_walk_search<E::kVec>(L, vbeg, vend, ae);
          }
          consumers_sync();
          alive = publish_draw(L, e, crank, csize, token, cert) && alive;
          if (!ms.go || !cert) flags |= SPEC_ROW_UNCERTIFIED;
          break;
        }
        if (token < 0 || !alive) error = true;
      }
    }
  }

  // ---------------------------------------------------------------- outputs
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
      if (a.row_info) a.row_info[b] = flags;
      if (error && a.err) {
        const int bit = *L.ring.abort ? SPEC_DERR_TIMEOUT
                        : ms.bad_token ? SPEC_DERR_TOKEN
                                       : SPEC_DERR_LOGITS;
        atomicOr(a.err, bit);
      }
    }
    if (warp == 0 && lane < K && a.q_at_d) {
      a.q_at_d[size_t(b) * K + lane] = ms.qd[lane];
      a.p_at_d[size_t(b) * K + lane] = ms.pd[lane];
    }
  }
  consumers_sync();  // the next row reuses every per-row buffer
}

// ------------------------------------------------------------------ kernel
template <class E>
__global__ void __launch_bounds__(kThreads, 2) verify_sample_kernel(const SampleArgs a, int ncl) {
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K, V = a.V, R = 2 * K + 1;
  const Layout L = make_layout(smem_raw, R);
  const int crank = int(cluster_ctarank()), csize = int(cluster_nctarank());
  const int cid = blockIdx.x / csize;
  int vbeg, vend;
  cta_slice(V / E::kVec, crank, csize, vbeg, vend);

  ring_xc_init(L.ring, L.xc, csize);
  __syncthreads();
  cluster_sync();  // every CTA's barriers are initialised before any remote arrive

  if (threadIdx.x >= kCons) {
    if (threadIdx.x == kCons) {
      uint32_t it = 0;
      for (int b = cid; b < a.B; b += ncl) {
        const T* tgt = static_cast<const T*>(a.target) + size_t(b) * (K + 1) * V;
        const T* drf = static_cast<const T*>(a.draft) + size_t(b) * K * V;
        auto rp = [&](int r) -> const T* {
          const int i = r >> 1;
          return (r & 1) ? drf + size_t(i) * V : tgt + size_t(i) * V;
        };
        it = produce_rows(L.ring, it, 2 * K, rp, vbeg, vend);
      }
    }
  } else {
    uint32_t it = 0, e = 0;
    for (int b = cid; b < a.B; b += ncl) verify_row<E>(a, L, b, vbeg, vend, crank, csize, it, e);
  }
  __syncthreads();
  cluster_sync();  // no CTA leaves while another may still address its shared memory
}

}  // namespace

int launch_verify_sample(const SampleLaunch& s) {
  SampleArgs a;
  a.target = s.target;
  a.draft = s.draft;
  a.tokens = s.tokens;
  a.uniforms = s.uniforms;
  a.B = s.B;
  a.K = s.K;
  a.V = s.V;
  const double C = 1.4426950408889634073599246810018921 / double(s.temperature);  // log2(e)/T
  a.c = float(C);
  a.Chi = float(C);
  a.Clo = float(C - double(a.Chi));
  const int kvec = (s.dtype == SPEC_BF16) ? 8 : 4;
  const int nvec = s.V / kvec;
  const int csize = pick_cluster(s.B, nvec);
  const int run = (nvec / csize) / kCons + 2;  // running-sum length per thread per row slice
  a.bd.ex2 = float(kEx2RelErrBound);
  a.bd.gamma1 = float((3.0 + run) * 5.9604644775390625e-8 * 1.01);
  a.bd.xbar = float(std::log2(double(s.V)) + 2.0);
  a.out_tokens = s.out_tokens;
  a.out_n = s.out_n;
  a.err = s.err;
  a.row_info = s.row_info;
  a.q_at_d = s.q_at_d;
  a.p_at_d = s.p_at_d;
  const size_t smem = sample_smem_bytes(2 * s.K + 1);
  cudaStream_t st = static_cast<cudaStream_t>(s.stream);
  if (s.dtype == SPEC_BF16)
    return launch_persistent(verify_sample_kernel<EBf16>, a, s.B, csize, smem, st);
  return launch_persistent(verify_sample_kernel<EF32>, a, s.B, csize, smem, st);
}

}  // namespace sv
