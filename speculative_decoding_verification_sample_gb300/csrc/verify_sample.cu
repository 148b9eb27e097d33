// Sampling-mode verification kernel (spec_verify_sample).
//
// Method ("aiengineeringfromscratch.com - Speculative decoding and EAGLE-3",
// "Variant: Leviathan rejection sampling" and Steps 1-3): draft token d_i is
// accepted iff p_i(d_i) <= 0 or u_i < min(1, q_i(d_i)/p_i(d_i)); at the first
// rejection j the correction is drawn from (q_j - p_j)+ (q_j if that mass is
// zero); after K acceptances a bonus token is drawn from q_K. The draw is the
// inverse CDF in token-index order with the single uniform u_K.
//
// GB300 mapping (dataflow engine, engine.cuh). Each batch row is cut into S
// vocabulary slices and goes through these stages, each a set of S slice
// tasks whose last finisher continues the row:
//   P1  softmax statistics (max, sum of exp2) of the slice of all 2K logit
//       rows (target and draft, positions 0..K-1), streamed from HBM;
//       finish: combine -> K accept tests -> first rejection j (warp ballot)
//   BS  (only when all K are accepted) statistics of target row K
//   SW  fp32 residual (q_j - p_j)+ (or q_K) over the slice of row j, re-read
//       while hot in L2; per 32-vector unit sums kept in the workspace;
//       finish: locate u_K * total mass slice -> unit -> entry, certify
//   FA  (rare) double-float row sums of the draw's rows
//   FB  (rare) double-float residual and unit sums; finish: certified search
// Only row j of the draft/target pair is ever re-read for the draw.
//
// Arithmetic. No fp64 arithmetic (GB300 runs fp64 at a small fraction of its
// fp32 rate): logits are widened to fp32, exponentials use the MUFU exp2 with
// an integer offset ceil(max * log2(e)/T), and sums a decision depends on are
// float pairs (df.cuh). A decision is taken from the fp32 path only when the
// uniform is farther from the threshold than twice a proven bound on that
// path's error; otherwise the FA/FB stages recompute it with double-float
// exponentials (relative error < 4e-12 per term) and the row is flagged in
// row_info. The output equals an exact-arithmetic evaluation except for rows
// flagged SPEC_ROW_UNCERTIFIED.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "../../include/specverify.h"
#include "common.cuh"
#include "df.cuh"
#include "engine.cuh"
#include "launch_util.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace sv {
namespace {

enum TaskType { kP1 = 1, kBS = 2, kSW = 3, kFA = 4, kFB = 5 };
enum { kAccept = 0, kReject = 1, kAmbiguous = 2, kInvalid = 3 };
constexpr int kModeResidual = 0, kModeQ = 1;  // RowState.mode

// ------------------------------------------------------------------ arguments
struct Bounds {
  float ex2;     // relative error bound of ex2.approx.ftz.f32 on [-126, 1]
  float gamma1;  // relative error bound of the per-thread fp32 summation of row sums
  float xbar;    // bound on sum_v q_v |x_v| used by the accept tests (log2 V + 2)
};

struct SampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  int B, K, V, S, nvec;
  float c;         // fl32(log2(e) / T)
  float Chi, Clo;  // log2(e) / T as a float pair
  Bounds bd;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  int32_t* row_info;
  float* q_at_d;
  float* p_at_d;
  Ws ws;
};

// ------------------------------------------------------------------ shared memory
struct Misc {
  int abort;
  int last;  // this CTA completed the stage of the current task's row
  int tok[kMaxK];
  float zt_d[kMaxK], zd_d[kMaxK], u[kMaxK + 1];
  int bad_token;
  int acc_state[kMaxK];
  float qd[kMaxK], pd[kMaxK];
  df wR[kCW];
  float wF[4][kCW];
  df wA[kCW], wB[kCW];
  int token, cert, found;
  df tstar, base;
  float E;
};

struct Smem {
  Ring ring;
  Misc* misc;
  float* wM;  // [2K+1][kCW]
  df* wS;     // [2K+1][kCW]
  int* wBad;  // [2K+1][kCW]
  float* rowKc;
  df* rowS;
  df* rowInv;
  int* rowOK;
  float* tab_hi;
  float* tab_lo;
};

__host__ __device__ inline size_t al(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <class F>
__host__ __device__ inline size_t carve(int R, F&& put) {
  size_t o = size_t(kStages) * kChunk;
  auto take = [&](size_t bytes, size_t a) {
    o = al(o, a);
    const size_t at = o;
    o += bytes;
    return at;
  };
  put(0, take(2 * kStages * 8, 8));
  put(1, take(kStages * sizeof(ChunkMeta), 16));
  put(2, take(kStages * sizeof(QTask), 16));
  put(3, take(sizeof(Misc), 16));
  put(4, take(size_t(R) * kCW * sizeof(df), 8));
  put(5, take(size_t(R) * sizeof(df) * 2, 8));
  put(6, take(size_t(R) * kCW * 8, 4));
  put(7, take(size_t(R) * 8, 4));
  put(8, take(256 * 8, 4));
  return al(o, 128);
}

__host__ __device__ inline size_t sample_smem_bytes(int R) { return carve(R, [](int, size_t) {}); }

__device__ inline Smem make_smem(uint8_t* base, int R) {
  Smem L;
  L.ring.buf = base;
  carve(R, [&](int id, size_t at) {
    uint8_t* p = base + at;
    switch (id) {
      case 0:
        L.ring.full = reinterpret_cast<uint64_t*>(p);
        L.ring.empty = L.ring.full + kStages;
        break;
      case 1:
        L.ring.meta = reinterpret_cast<ChunkMeta*>(p);
        break;
      case 2:
        L.ring.ttab = reinterpret_cast<QTask*>(p);
        break;
      case 3:
        L.misc = reinterpret_cast<Misc*>(p);
        L.ring.abort = &L.misc->abort;
        break;
      case 4:
        L.wS = reinterpret_cast<df*>(p);
        break;
      case 5:
        L.rowS = reinterpret_cast<df*>(p);
        L.rowInv = L.rowS + R;
        break;
      case 6:
        L.wM = reinterpret_cast<float*>(p);
        L.wBad = reinterpret_cast<int*>(L.wM + R * kCW);
        break;
      case 7:
        L.rowKc = reinterpret_cast<float*>(p);
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

// ------------------------------------------------------------------ statistics
// Per-thread running max M, integer offset Kc = ceil(M c) and S = sum exp2(z c - Kc).
template <class E>
struct StatOp {
  float c, M, Kc, S;
  int bad;
  __device__ __forceinline__ void begin() {
    M = -INFINITY;
    Kc = -INFINITY;
    S = 0.0f;
    bad = 0;
  }
  // The vectors i = tid, tid + kCons, ... < cnt of one ring stage (at most
  // kPer per thread): loaded together, one running-maximum update per stage,
  // then the exponentials, so the loads and MUFU operations overlap.
  __device__ __forceinline__ void chunk(const uint4* buf, int cnt, int tid) {
    constexpr int kPer = kChunk / 16 / kCons;
    uint4 v[kPer];
    float vm = -INFINITY;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (tid + k * kCons < cnt) {
        v[k] = buf[tid + k * kCons];
        vm = max_nan(vm, E::vmax(v[k]));
      }
    }
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
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (tid + k * kCons < cnt) {
        float z[E::kVec];
        E::unpack(v[k], z);
        float e[E::kVec];
#pragma unroll
        for (int j = 0; j < E::kVec; ++j) e[j] = ex2_approx(__fmaf_rn(z[j], c, -Kc));
#pragma unroll
        for (int w = 1; w < E::kVec; w <<= 1)
#pragma unroll
          for (int j = 0; j < E::kVec; j += 2 * w) e[j] = __fadd_rn(e[j], e[j + w]);
        S = __fadd_rn(S, e[0]);
      }
    }
  }
  // warp partial of row r into smem
  __device__ void end_row(const Smem& L, int r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float Mw = warp_max_f(M);
    df s{0.f, 0.f};
    if (S != 0.0f) s.hi = __fmul_rn(S, pow2i(__fsub_rn(Kc, offset_of(Mw, c))));
    s = df_warp_sum(s);
    const int anybad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      L.wM[r * kCW + warp] = Mw;
      L.wS[r * kCW + warp] = s;
      L.wBad[r * kCW + warp] = anybad;
    }
  }
};

// CTA partial (M, S.hi, S.lo, bad) of rows [0, nrows) into out[4r..4r+3].
__device__ void stats_to_global(const Smem& L, int nrows, float c, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < nrows; r += kCW) {
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
      float* o = out + 4 * r;
      o[0] = Mc;
      o[1] = s.hi;
      o[2] = s.lo;
      o[3] = __int_as_float(bad);
    }
  }
}

// Row statistics (into smem slot rs) from the S slice partials of row r at
// float offset 4r of each slice's part block; same order everywhere.
__device__ void stats_combine(const SampleArgs& a, const Smem& L, int b, int r, int rs) {
  float M = -INFINITY;
  int bad = 0;
  for (int s = 0; s < a.S; ++s) {
    const float* p = a.ws.part(b, s) + 4 * r;
    M = fmaxf(M, ld_cg_f(p));
    bad |= __float_as_int(ld_cg_f(p + 3));
  }
  const float Kc = offset_of(M, a.c);
  df S{0.f, 0.f};
  for (int s = 0; s < a.S; ++s) {
    const float* p = a.ws.part(b, s) + 4 * r;
    const float sh = ld_cg_f(p + 1);
    if (sh != 0.0f) {
      const float sc = pow2i(__fsub_rn(offset_of(ld_cg_f(p), a.c), Kc));
      S = df_add(S, df{__fmul_rn(sh, sc), __fmul_rn(ld_cg_f(p + 2), sc)});
    }
  }
  const bool ok = !bad && isfinite(M) && fabsf(Kc) < 4194304.0f && S.hi > 0.0f && isfinite(S.hi);
  L.rowKc[rs] = Kc;
  L.rowS[rs] = S;
  L.rowInv[rs] = ok ? df_recip(S) : df{0.f, 0.f};
  L.rowOK[rs] = ok ? 1 : 0;
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

// Relative error bound of one normalised double-float term: the exponential
// (< 4e-13), its argument (< 2^-46 (|z C| + |Kc|), offsets below 2^22 by the
// row checks), the normaliser sum and reciprocal; kept above their total.
constexpr float kAccRho = 4e-12f;

// Upper bound on the sum of the computed fp32 probabilities of a row.
constexpr float kQmax = 1.001f;

__device__ inline void load_table(const Smem& L) {
  for (int i = threadIdx.x; i < 256; i += kCons) {
    L.tab_hi[i] = kExp2Tab.hi[i];
    L.tab_lo[i] = kExp2Tab.lo[i];
  }
}

// ------------------------------------------------------------------ draw entries
// fp32 path: r = max(0, q - p), q = exp2(z c - Kq) * Rq (r = q when tp is
// null). aq / ap accumulate sum q x and sum p x (x the exponent argument,
// clamped at -1e4 so that masked logits add 0), from which the error bound
// of the sweep follows.
template <class E>
struct FastEntries {
  const uint4* tq;
  const uint4* tp;
  float c, Kq, Rq, Kp, Rp;
  __device__ __forceinline__ float run(const uint4& vq, const uint4& vp, float (&r)[E::kVec],
                                       float& aq, float& ap) const {
    float zq[E::kVec], zp[E::kVec];
    E::unpack(vq, zq);
    if (tp) E::unpack(vp, zp);
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      const float xa = __fmaf_rn(zq[k], c, -Kq);
      const float q = __fmul_rn(ex2_approx(xa), Rq);
      aq = __fmaf_rn(q, fmaxf(xa, -1.0e4f), aq);
      if (tp) {
        const float xb = __fmaf_rn(zp[k], c, -Kp);
        const float p = __fmul_rn(ex2_approx(xb), Rp);
        ap = __fmaf_rn(p, fmaxf(xb, -1.0e4f), ap);
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
  __device__ __forceinline__ df entries(int vi, df (&rd)[E::kVec]) const {
    float r[E::kVec];
    float a0 = 0.f, a1 = 0.f;
    const uint4 vq = ldg_nc_v4(tq + vi);
    const uint4 vp = tp ? ldg_nc_v4(tp + vi) : vq;
    const float vs = run(vq, vp, r, a0, a1);
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
  df Iq, Ip;
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
    float a0 = 0.f, a1 = 0.f;
    const uint4 vq = ldg_nc_v4(tq + vi);
    const uint4 vp = tp ? ldg_nc_v4(tp + vi) : vq;
    return run(vq, vp, rd, a0, a1);
  }
};

// ------------------------------------------------------------------ helpers
template <class E>
struct RowPtrs {
  const typename E::T* tgt;
  const typename E::T* drf;
};

template <class E>
__device__ __forceinline__ RowPtrs<E> row_ptrs(const SampleArgs& a, int b) {
  using T = typename E::T;
  return {static_cast<const T*>(a.target) + size_t(b) * (a.K + 1) * a.V,
          static_cast<const T*>(a.draft) + size_t(b) * a.K * a.V};
}

// Consumers: block sum of a per-thread pair and four floats (thread 0 gets
// the totals).
__device__ void cta_reduce(Misc& ms, df& r, float (&f)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  r = df_warp_sum(r);
#pragma unroll
  for (int j = 0; j < 4; ++j) f[j] = warp_sum_f(f[j]);
  if (lane == 0) {
    ms.wR[warp] = r;
#pragma unroll
    for (int j = 0; j < 4; ++j) ms.wF[j][warp] = f[j];
  }
  consumers_sync();
  if (threadIdx.x == 0) {
    r = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = 0.f;
    for (int w = 0; w < kCW; ++w) {
      r = df_add(r, ms.wR[w]);
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] += ms.wF[j][w];
    }
  }
}

// Consumers: publish the task's partials (already stored) and arrive on the
// row's stage counter. Returns true in every thread when this CTA completed
// the stage (then it must continue the row).
__device__ bool arrive_row(const SampleArgs& a, Misc& ms, int b) {
  __threadfence();
  consumers_sync();
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(&a.ws.row_cnt()[b], 1u);
    const int last = (old == uint32_t(a.S) - 1);
    if (last) {
      a.ws.row_cnt()[b] = 0;  // the next stage counts from zero
      __threadfence();
    }
    ms.last = last;
  }
  consumers_sync();
  return ms.last != 0;
}

__device__ void write_outputs(const SampleArgs& a, const Misc& ms, int b, int n, int token,
                              int flags, bool error) {
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
    if (a.row_info) a.row_info[b] = flags;
  }
  __threadfence();
  consumers_sync();
  if (threadIdx.x == 0) atomicAdd(&a.ws.hdr()->rows_done, 1u);
}

// Locate the slice, then the 32-vector unit, holding t, then the entry (warp 0
// walks the unit). ms.token / ms.cert receive the result; certified iff both
// boundaries of the drawn entry are farther than 2E from t.
template <class E, class Entries>
__device__ void search_draw(const SampleArgs& a, Misc& ms, int b, const Entries& ent) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const df t = ms.tstar;
    // slice: lanes scan 32 slices at a time; the first slice with mass whose
    // end passes t, else the last slice with mass (rounding fallback)
    int ss = -1;
    df pre_s{0.f, 0.f};
    {
      df sbase{0.f, 0.f};
      for (int s0 = 0; s0 < a.S; s0 += 32) {
        const int s = s0 + lane;
        df x{0.f, 0.f};
        if (s < a.S) {
          const float* p = a.ws.part(b, s);
          x = df{ld_cg_f(p), ld_cg_f(p + 1)};
        }
        df inc = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const df y = df_shfl_up(inc, o);
          if (lane >= o) inc = df_add(inc, y);
        }
        const df lo = df_add(sbase, df_sub(inc, x));
        const unsigned hm = __ballot_sync(0xffffffffu, x.hi > 0.0f && df_gt(df_add(lo, x), t));
        const unsigned pm = __ballot_sync(0xffffffffu, x.hi > 0.0f);
        if (hm) {
          const int l = __ffs(int(hm)) - 1;
          ss = s0 + l;
          pre_s = df_shfl(lo, l);
          break;
        }
        if (pm) {
          const int l = 31 - __clz(int(pm));
          ss = s0 + l;
          pre_s = df_shfl(lo, l);
        }
        sbase = df_add(sbase, df_shfl(inc, 31));
      }
    }
    int token = -1;
    df tlo = pre_s, thi = pre_s;
    if (ss >= 0) {
      int v0, v1;
      slice_range(a.nvec, a.S, ss, v0, v1);
      const int nu = (v1 - v0 + 31) / 32;
      // unit: lanes scan 32 units at a time
      const float2* up = a.ws.units(b, ss);
      int us = -1;
      df ubase = pre_s, ubase_s = pre_s;
      for (int u0 = 0; u0 < nu && us < 0; u0 += 32) {
        const int u = u0 + lane;
        df x{0.f, 0.f};
        if (u < nu) x = df{__ldcg(&up[u].x), __ldcg(&up[u].y)};
        df inc = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const df y = df_shfl_up(inc, o);
          if (lane >= o) inc = df_add(inc, y);
        }
        const df lo = df_add(ubase, df_sub(inc, x));
        const bool hit = x.hi > 0.0f && df_gt(df_add(lo, x), t);
        const unsigned hm = __ballot_sync(0xffffffffu, hit);
        const unsigned pm = __ballot_sync(0xffffffffu, u < nu && x.hi > 0.0f);
        if (hm) {
          const int l = __ffs(int(hm)) - 1;
          us = u0 + l;
          ubase_s = df_shfl(lo, l);
        } else if (pm) {
          const int l = 31 - __clz(int(pm));
          ubase_s = df_shfl(lo, l);  // last unit with mass so far (rounding fallback)
          us = -(u0 + l) - 2;
        }
        ubase = df_add(ubase, df_shfl(inc, 31));
      }
      if (us < -1) us = -us - 2;
      if (us >= 0) {
        // entries of the unit's 32 vectors, lane-minor
        const int vi = v0 + us * 32 + lane;
        df r[E::kVec];
        df vs{0.f, 0.f};
        if (vi < v1) {
          vs = ent.entries(vi, r);
        } else {
#pragma unroll
          for (int k = 0; k < E::kVec; ++k) r[k] = {0.f, 0.f};
        }
        df inc = vs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const df y = df_shfl_up(inc, o);
          if (lane >= o) inc = df_add(inc, y);
        }
        df c0 = df_add(ubase_s, df_sub(inc, vs));
        int tk = -1, lk = -1;
        df lo{0.f, 0.f}, hi{0.f, 0.f}, l0{0.f, 0.f}, l1{0.f, 0.f};
#pragma unroll
        for (int k = 0; k < E::kVec; ++k) {
          const df c1 = df_add(c0, r[k]);
          if (r[k].hi > 0.0f) {
            lk = vi * E::kVec + k;
            l0 = c0;
            l1 = c1;
            if (tk < 0 && df_gt(c1, t)) {
              tk = vi * E::kVec + k;
              lo = c0;
              hi = c1;
            }
          }
          c0 = c1;
        }
        const unsigned hm = __ballot_sync(0xffffffffu, tk >= 0);
        const unsigned pm = __ballot_sync(0xffffffffu, lk >= 0);
        if (hm) {
          const int l = __ffs(int(hm)) - 1;
          token = __shfl_sync(0xffffffffu, tk, l);
          tlo = df_shfl(lo, l);
          thi = df_shfl(hi, l);
        } else if (pm) {
          const int l = 31 - __clz(int(pm));
          token = __shfl_sync(0xffffffffu, lk, l);
          tlo = df_shfl(l0, l);
          thi = df_shfl(l1, l);
        }
      }
    }
    if (lane == 0) {
      const float m1 = df_sub(t, tlo).hi, m2 = df_sub(thi, t).hi;
      ms.token = token;
      ms.cert = (token >= 0 && fminf(m1, m2) > 2.02f * ms.E) ? 1 : 0;
    }
  }
  consumers_sync();
}

// ------------------------------------------------------------------ stage finishers
// P1 complete: statistics of the 2K rows, accept tests, first rejection.
template <class E>
__device__ void finish_p1(const SampleArgs& a, const Smem& L, int b) {
  Misc& ms = *L.misc;
  const int K = a.K, V = a.V, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const RowPtrs<E> rp = row_ptrs<E>(a, b);
  for (int r = tid; r < 2 * K; r += kCons) stats_combine(a, L, b, r, r);
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
        ms.zt_d[lane] = E::load(rp.tgt + size_t(lane) * V, d);
        ms.zd_d[lane] = E::load(rp.drf + size_t(lane) * V, d);
      }
    }
    if (lane <= K) ms.u[lane] = a.uniforms[size_t(b) * (K + 1) + lane];
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) ms.bad_token = bad;
  }
  consumers_sync();
  const float c = a.c;
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
        // arguments (with the fp32 temperature constant), both row sums and
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
    if (a.q_at_d) {
      a.q_at_d[size_t(b) * K + i] = qd;
      a.p_at_d[size_t(b) * K + i] = pd;
    }
  }
  consumers_sync();

  int flags = 0, n = 0;
  bool error = ms.bad_token != 0;
  while (!error) {
    int i = n;
    while (i < K && ms.acc_state[i] == kAccept) ++i;
    n = i;
    if (i == K) break;
    const int st = ms.acc_state[i];
    if (st == kInvalid) {
      error = true;
      break;
    }
    if (st == kReject) break;
    // ambiguous: decide with accurate sums of target and draft row i over the
    // whole vocabulary (this CTA alone; probability ~1e-6 per test)
    flags |= SPEC_ROW_ACCEPT_REFINED;
    load_table(L);
    consumers_sync();
    df s0{0.f, 0.f}, s1{0.f, 0.f};
    {
      const uint4* p0 = reinterpret_cast<const uint4*>(rp.tgt + size_t(i) * V);
      const uint4* p1 = reinterpret_cast<const uint4*>(rp.drf + size_t(i) * V);
      const float K0 = L.rowKc[2 * i], K1 = L.rowKc[2 * i + 1];
      for (int vi = tid; vi < a.nvec; vi += kCons) {
        float z[E::kVec];
        E::unpack(ldg_nc_v4(p0 + vi), z);
#pragma unroll
        for (int k = 0; k < E::kVec; ++k)
          s0 = df_add(s0, acc_elem(z[k], a.Chi, a.Clo, K0, L.tab_hi, L.tab_lo));
        E::unpack(ldg_nc_v4(p1 + vi), z);
#pragma unroll
        for (int k = 0; k < E::kVec; ++k)
          s1 = df_add(s1, acc_elem(z[k], a.Chi, a.Clo, K1, L.tab_hi, L.tab_lo));
      }
      s0 = df_warp_sum(s0);
      s1 = df_warp_sum(s1);
      if (lane == 0) {
        ms.wA[warp] = s0;
        ms.wB[warp] = s1;
      }
      consumers_sync();
      s0 = s1 = {0.f, 0.f};
      for (int w = 0; w < kCW; ++w) {
        s0 = df_add(s0, ms.wA[w]);
        s1 = df_add(s1, ms.wB[w]);
      }
    }
    // ratio = 2^((zt C - Kt) - (zd C - Kd)) * S_d / S_t in pair arithmetic
    const float zt = ms.zt_d[i], zd = ms.zd_d[i], u = ms.u[i];
    const df xt =
        df_add_f(df_add(two_prod(zt, a.Chi), df{__fmul_rn(zt, a.Clo), 0.f}), -L.rowKc[2 * i]);
    const df xd =
        df_add_f(df_add(two_prod(zd, a.Chi), df{__fmul_rn(zd, a.Clo), 0.f}), -L.rowKc[2 * i + 1]);
    const df ar = df_sub(xt, xd);
    bool acc;
    if (ar.hi >= 127.0f) {
      acc = true;
    } else if (ar.hi < -126.0f) {
      acc = false;  // ratio < 2^-100 < u (u > 0 here)
    } else {
      const df ratio = df_mul(df_mul(df_exp2(ar.hi, ar.lo, L.tab_hi, L.tab_lo), s1), df_recip(s0));
      acc = (ratio.hi >= 1.0f) || df_gt(ratio, df{u, 0.f});
      if (fabsf(__fsub_rn(u, fminf(1.0f, ratio.hi))) <= 1e-10f * ratio.hi) flags |= SPEC_ROW_UNCERTIFIED;
    }
    consumers_sync();
    if (!acc) break;
    if (tid == 0) ms.acc_state[i] = kAccept;
    consumers_sync();
    n = i + 1;
  }
  if (error) {
    if (tid == 0 && a.err) atomicOr(a.err, ms.bad_token ? SPEC_DERR_TOKEN : SPEC_DERR_LOGITS);
    write_outputs(a, ms, b, n, -1, flags, true);
    return;
  }
  if (tid == 0) {
    RowState* st = a.ws.rowstate(b);
    st->n = n;
    st->flags = flags;
    st->err = 0;
    if (n < K) {
      st->mode = kModeResidual;
      st->Kq = L.rowKc[2 * n];
      st->Rq = L.rowInv[2 * n].hi;
      st->Kp = L.rowKc[2 * n + 1];
      st->Rp = L.rowInv[2 * n + 1].hi;
    } else {
      st->mode = kModeQ;
    }
    __threadfence();
    enqueue_row_stage(a.ws, n < K ? kSW : kBS, b, a.S, n);
  }
}

// ------------------------------------------------------------------ kernel
template <class E>
__global__ void __launch_bounds__(kThreads, 2) verify_sample_kernel(const SampleArgs a) {
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K, R = 2 * K + 1;
  const Smem L = make_smem(smem_raw, R);
  Misc& ms = *L.misc;
  ring_init(L.ring);
  __syncthreads();

  if (threadIdx.x >= kCons) {
    // ------------------------------------------------ producer
    if (threadIdx.x == kCons) {
      uint32_t it = 0, nt = 0;
      uint64_t idle_t0 = 0;
      int64_t pending = -1;
      WsHeader* h = a.ws.hdr();
      while (!*L.ring.abort && !ld_volatile_u32(&h->abort)) {
        QTask t;
        bool exhausted;
        if (!fetch_task(a.ws, kP1, t, exhausted, pending)) {
          if (!producer_idle(a.ws, exhausted, idle_t0)) break;
          continue;
        }
        idle_t0 = 0;
        const RowPtrs<E> rp = row_ptrs<E>(a, t.b);
        int v0, v1;
        slice_range(a.nvec, a.S, t.s, v0, v1);
        const char* rows[2 * kMaxK];
        int nrows = 0;
        bool paired = false;
        if (t.type == kP1) {
          for (int i = 0; i < K; ++i) {
            rows[nrows++] = reinterpret_cast<const char*>(rp.tgt + size_t(i) * a.V);
            rows[nrows++] = reinterpret_cast<const char*>(rp.drf + size_t(i) * a.V);
          }
        } else if (t.type == kBS) {
          rows[nrows++] = reinterpret_cast<const char*>(rp.tgt + size_t(K) * a.V);
        } else {
          const int n = t.aux & 0xff, mode = t.aux >> 8;
          const int j = n;  // row j (j = K for the bonus draw)
          rows[nrows++] = reinterpret_cast<const char*>(rp.tgt + size_t(j) * a.V);
          if (mode == kModeResidual && n < K) {
            rows[nrows++] = reinterpret_cast<const char*>(rp.drf + size_t(j) * a.V);
            paired = true;
          }
        }
        if (!produce_task(L.ring, it, nt, t, rows, nrows, paired, v0, v1)) break;
      }
      produce_end(L.ring, it);
    }
  } else {
    // ------------------------------------------------ consumers
    uint32_t it = 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    while (true) {
      if (!wait_stage(L.ring, it)) break;
      const ChunkMeta m0 = L.ring.meta[it % kStages];
      if (m0.slot < 0) break;
      const QTask t = L.ring.ttab[m0.slot];
      const int b = t.b, s = t.s;
      const RowPtrs<E> rp = row_ptrs<E>(a, b);
      int v0, v1;
      slice_range(a.nvec, a.S, s, v0, v1);
      if (t.type == kP1 || t.type == kBS) {
        // ---------------- statistics of the slice of every row of the task
        StatOp<E> op;
        op.c = a.c;
        op.begin();
        for (;;) {
          const ChunkMeta m = L.ring.meta[it % kStages];
          const uint4* buf = stage_data(L.ring, it);
          op.chunk(buf, m.c1 - m.c0, tid);
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
        const int nrows = (t.type == kP1) ? 2 * K : 1;
        stats_to_global(L, nrows, a.c, a.ws.part(b, s));
        if (arrive_row(a, ms, b)) {
          if (t.type == kP1) {
            finish_p1<E>(a, L, b);
          } else {
            // bonus statistics of target row K -> its draw
            if (tid == 0) {
              stats_combine(a, L, b, 0, 2 * K);
              RowState* st = a.ws.rowstate(b);
              if (!L.rowOK[2 * K]) {
                st->err = 1;
              } else {
                st->Kq = L.rowKc[2 * K];
                st->Rq = L.rowInv[2 * K].hi;
              }
            }
            consumers_sync();
            const RowState* st = a.ws.rowstate(b);
            if (ld_cg_i(&st->err)) {
              if (warp == 1 && lane < K) ms.tok[lane] = a.tokens[size_t(b) * K + lane];
              consumers_sync();
              if (tid == 0 && a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
              write_outputs(a, ms, b, K, -1, ld_cg_i(&st->flags), true);
            } else if (tid == 0) {
              __threadfence();
              enqueue_row_stage(a.ws, kSW, b, a.S, K | (kModeQ << 8));
            }
          }
        }
        consumers_sync();
        continue;
      }
      // ------------------------------------------------ draw stages
      const RowState* stp = a.ws.rowstate(b);
      const int n = t.aux & 0xff, mode = t.aux >> 8;
      const bool pair = (mode == kModeResidual && n < K);
      const int jrow = n;
      const uint4* vq = reinterpret_cast<const uint4*>(rp.tgt + size_t(jrow) * a.V);
      const uint4* vp = pair ? reinterpret_cast<const uint4*>(rp.drf + size_t(jrow) * a.V) : nullptr;
      if (t.type == kSW) {
        FastEntries<E> fe;
        fe.tq = vq;
        fe.tp = vp;
        fe.c = a.c;
        fe.Kq = ld_cg_f(&stp->Kq);
        fe.Rq = ld_cg_f(&stp->Rq);
        fe.Kp = pair ? ld_cg_f(&stp->Kp) : 0.f;
        fe.Rp = pair ? ld_cg_f(&stp->Rp) : 0.f;
        constexpr int kPer = kChunk / 16 / kCons;
        float accf = 0.f, Aq = 0.f, Ap = 0.f;
        float2* units = a.ws.units(b, s);
        for (;;) {
          const ChunkMeta m = L.ring.meta[it % kStages];
          const uint4* bq = stage_data(L.ring, it);
          const uint4* bp = bq;
          uint32_t it2 = it;
          if (pair) {
            if (!wait_stage(L.ring, it + 1)) break;
            bp = stage_data(L.ring, it + 1);
            it2 = it + 1;
          }
          const int cnt = m.c1 - m.c0;
          // unit u of this stage = vectors [32u, 32u + 32): warp w takes units
          // w, w + 8, ...; every lane one vector pair of each
          float vs[kPer];
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int i = warp * 32 + k * kCons + lane;
            vs[k] = 0.f;
            if (i < cnt) {
              float r[E::kVec];
              vs[k] = fe.run(bq[i], bp[i], r, Aq, Ap);
            }
          }
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int i0 = warp * 32 + k * kCons;
            if (i0 < cnt) {
              const float us = warp_sum_f(vs[k]);
              if (lane == 0) units[(m.c0 - v0 + i0) / 32] = make_float2(us, 0.f);
            }
            accf = __fadd_rn(accf, vs[k]);
          }
          const bool lastc = L.ring.meta[it2 % kStages].last != 0;
          release_stage(L.ring, it);
          if (pair) release_stage(L.ring, it2);
          it = it2 + 1;
          if (lastc) break;
          if (!wait_stage(L.ring, it)) break;
        }
        df acc{accf, 0.f};
        float f4[4] = {Aq, Ap, 0.f, 0.f};
        cta_reduce(ms, acc, f4);
        if (tid == 0) {
          float* o = a.ws.part(b, s);
          o[0] = acc.hi;
          o[1] = acc.lo;
          o[2] = f4[0];
          o[3] = f4[1];
        }
        if (arrive_row(a, ms, b)) {
          // ---------------- fp32 draw: bound, locate, certify
          if (tid == 0) {
            df Sr{0.f, 0.f};
            float Aqt = 0.f, Apt = 0.f;
            for (int q = 0; q < a.S; ++q) {
              const float* p = a.ws.part(b, q);
              Sr = df_add(Sr, df{ld_cg_f(p), ld_cg_f(p + 1)});
              Aqt += ld_cg_f(p + 2);
              Apt += ld_cg_f(p + 3);
            }
            // Error bound (probability units) of the fp32 sweep. Per term,
            // relative: exp2 (ex2), argument rounding and the fp32
            // temperature constant (ln2 u |x| each), 1/S and the product
            // (3u), and the row sum behind 1/S (ex2 + ln2 u sum q|x| +
            // gamma1); summed with weights q (resp. p), whose sum is at most
            // kQmax. sum q|x| <= kQmax/2 - sum q x, since x <= 1/4 (the offset
            // is ceil of the rounded max * c, below 2^22 in magnitude).
            // Rounding of the unit, slice and row sums adds 16 u Sr.
            auto side = [&](float A) {
              const float absx = 1.01f * fmaxf(0.0f, -A) + 0.5f * kQmax;
              return 1.05f * (kQmax * (2.0f * a.bd.ex2 + 3.0f * kU + a.bd.gamma1 + 4.0f * kLn2f * kU) +
                              4.0f * kLn2f * kU * absx);
            };
            const float E = side(Aqt) + (pair ? side(Apt) : 0.f) + 16.0f * kU * Sr.hi + 1e-30f;
            ms.E = E;
            ms.tstar = df_mul_f(Sr, a.uniforms[size_t(b) * (K + 1) + K]);
            ms.found = (Sr.hi > 2.0f * E) ? 1 : 0;
          }
          consumers_sync();
          if (ms.found) search_draw<E>(a, ms, b, fe);
          const int flags = ld_cg_i(&stp->flags);
          if (ms.found && ms.cert) {
            if (warp == 1 && lane < K) ms.tok[lane] = a.tokens[size_t(b) * K + lane];
            consumers_sync();
            write_outputs(a, ms, b, n, ms.token, flags, false);
          } else if (tid == 0) {
            RowState* st = a.ws.rowstate(b);
            st->flags = flags | SPEC_ROW_SAMPLE_REFINED;
            __threadfence();
            enqueue_row_stage(a.ws, kFA, b, a.S, t.aux);
          }
        }
        consumers_sync();
        continue;
      }
      // ---------------- double-float stages (rare)
      load_table(L);
      consumers_sync();
      if (t.type == kFA) {
        df s0{0.f, 0.f}, s1{0.f, 0.f};
        const float K0 = ld_cg_f(&stp->Kq), K1 = pair ? ld_cg_f(&stp->Kp) : 0.f;
        for (;;) {
          const ChunkMeta m = L.ring.meta[it % kStages];
          const uint4* buf = stage_data(L.ring, it);
          const float Kr = (m.r == 0) ? K0 : K1;
          df acc{0.f, 0.f};
          for (int i = tid; i < m.c1 - m.c0; i += kCons) {
            float z[E::kVec];
            E::unpack(buf[i], z);
#pragma unroll
            for (int k = 0; k < E::kVec; ++k)
              acc = df_add(acc, acc_elem(z[k], a.Chi, a.Clo, Kr, L.tab_hi, L.tab_lo));
          }
          if (m.r == 0) s0 = df_add(s0, acc);
          else s1 = df_add(s1, acc);
          release_stage(L.ring, it);
          ++it;
          if (m.last) break;
          if (!wait_stage(L.ring, it)) break;
        }
        s0 = df_warp_sum(s0);
        s1 = df_warp_sum(s1);
        if (lane == 0) {
          ms.wA[warp] = s0;
          ms.wB[warp] = s1;
        }
        consumers_sync();
        if (tid == 0) {
          df t0{0.f, 0.f}, t1{0.f, 0.f};
          for (int w = 0; w < kCW; ++w) {
            t0 = df_add(t0, ms.wA[w]);
            t1 = df_add(t1, ms.wB[w]);
          }
          float* o = a.ws.part(b, s);
          o[0] = t0.hi;
          o[1] = t0.lo;
          o[2] = t1.hi;
          o[3] = t1.lo;
        }
        if (arrive_row(a, ms, b) && tid == 0) {
          df S0{0.f, 0.f}, S1{0.f, 0.f};
          for (int q = 0; q < a.S; ++q) {
            const float* p = a.ws.part(b, q);
            S0 = df_add(S0, df{ld_cg_f(p), ld_cg_f(p + 1)});
            S1 = df_add(S1, df{ld_cg_f(p + 2), ld_cg_f(p + 3)});
          }
          RowState* st = a.ws.rowstate(b);
          const df I0 = df_recip(S0);
          st->Iq_hi = I0.hi;
          st->Iq_lo = I0.lo;
          if (pair) {
            const df I1 = df_recip(S1);
            st->Ip_hi = I1.hi;
            st->Ip_lo = I1.lo;
          }
          __threadfence();
          enqueue_row_stage(a.ws, kFB, b, a.S, t.aux);
        }
        consumers_sync();
        continue;
      }
      // kFB: double-float residual sums and unit sums
      AccEntries<E> ae;
      ae.tq = vq;
      ae.tp = vp;
      ae.Chi = a.Chi;
      ae.Clo = a.Clo;
      ae.Kq = ld_cg_f(&stp->Kq);
      ae.Kp = pair ? ld_cg_f(&stp->Kp) : 0.f;
      ae.Iq = df{ld_cg_f(&stp->Iq_hi), ld_cg_f(&stp->Iq_lo)};
      ae.Ip = pair ? df{ld_cg_f(&stp->Ip_hi), ld_cg_f(&stp->Ip_lo)} : df{0.f, 0.f};
      ae.th = L.tab_hi;
      ae.tl = L.tab_lo;
      {
        df acc{0.f, 0.f};
        float Q = 0.f, P = 0.f;
        float2* units = a.ws.units(b, s);
        for (;;) {
          const ChunkMeta m = L.ring.meta[it % kStages];
          const uint4* bq = stage_data(L.ring, it);
          const uint4* bp = bq;
          uint32_t it2 = it;
          if (pair) {
            if (!wait_stage(L.ring, it + 1)) break;
            bp = stage_data(L.ring, it + 1);
            it2 = it + 1;
          }
          const int cnt = m.c1 - m.c0;
          for (int i0 = warp * 32; i0 < cnt; i0 += kCons) {
            const int i = i0 + lane;
            df vs{0.f, 0.f};
            if (i < cnt) {
              df r[E::kVec];
              vs = ae.run(bq[i], bp[i], r, Q, P);
              acc = df_add(acc, vs);
            }
            const df us = df_warp_sum(vs);
            if (lane == 0) units[(m.c0 - v0 + i0) / 32] = make_float2(us.hi, us.lo);
          }
          const bool lastc = L.ring.meta[it2 % kStages].last != 0;
          release_stage(L.ring, it);
          if (pair) release_stage(L.ring, it2);
          it = it2 + 1;
          if (lastc) break;
          if (!wait_stage(L.ring, it)) break;
        }
        float f4[4] = {Q, P, 0.f, 0.f};
        cta_reduce(ms, acc, f4);
        if (tid == 0) {
          float* o = a.ws.part(b, s);
          o[0] = acc.hi;
          o[1] = acc.lo;
          o[2] = f4[0];
          o[3] = f4[1];
        }
      }
      if (arrive_row(a, ms, b)) {
        if (tid == 0) {
          df Sr{0.f, 0.f};
          float Qt = 0.f, Pt = 0.f;
          for (int q = 0; q < a.S; ++q) {
            const float* p = a.ws.part(b, q);
            Sr = df_add(Sr, df{ld_cg_f(p), ld_cg_f(p + 1)});
            Qt += ld_cg_f(p + 2);
            Pt += ld_cg_f(p + 3);
          }
          ms.E = kAccRho * (Qt + Pt) + 1e-14f * Sr.hi + 1e-36f;
          ms.tstar = df_mul_f(Sr, a.uniforms[size_t(b) * (K + 1) + K]);
          ms.found = (Sr.hi > 0.0f) ? 1 : (pair ? 2 : 0);  // 2: zero residual mass
        }
        consumers_sync();
        const int flags = ld_cg_i(&stp->flags);
        if (ms.found == 2) {
          // zero residual mass: the draw uses q_j itself
          if (tid == 0) {
            RowState* st = a.ws.rowstate(b);
            st->flags = flags | SPEC_ROW_ZERO_RESIDUAL;
            __threadfence();
            enqueue_row_stage(a.ws, kFB, b, a.S, n | (kModeQ << 8));
          }
        } else {
          if (ms.found == 1) search_draw<E>(a, ms, b, ae);
          if (warp == 1 && lane < K) ms.tok[lane] = a.tokens[size_t(b) * K + lane];
          consumers_sync();
          const int tokn = ms.found == 1 ? ms.token : -1;
          int fl = flags;
          if (!(ms.found == 1 && ms.cert)) fl |= SPEC_ROW_UNCERTIFIED;
          if (tokn < 0 && tid == 0 && a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
          write_outputs(a, ms, b, n, tokn, fl, tokn < 0);
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

}  // namespace

// ------------------------------------------------------------------ host side
namespace {

WsLayout sample_layout(int B, int K, int V, int dtype) {
  const int kvec = (dtype == SPEC_BF16) ? 8 : 4;
  const int nvec = V / kvec;
  const int S = slices_for(nvec, B);
  const int maxslice = (nvec + S - 1) / S;
  const int ustride = (maxslice + 31) / 32 + 1;
  const int part = (8 * K > 8) ? 8 * K : 8;
  return ws_layout(B, S, part, ustride, 5);
}

}  // namespace

size_t sample_workspace_bytes(int B, int K, int V, int dtype) {
  return sample_layout(B, K, V, dtype).total;
}

int launch_verify_sample(const SampleLaunch& s) {
  SampleArgs a;
  a.target = s.target;
  a.draft = s.draft;
  a.tokens = s.tokens;
  a.uniforms = s.uniforms;
  a.B = s.B;
  a.K = s.K;
  a.V = s.V;
  const int kvec = (s.dtype == SPEC_BF16) ? 8 : 4;
  a.nvec = s.V / kvec;
  const WsLayout wl = sample_layout(s.B, s.K, s.V, s.dtype);
  a.S = wl.S;
  a.ws.base = static_cast<uint8_t*>(s.workspace);
  a.ws.L = wl;
  const double C = 1.4426950408889634073599246810018921 / double(s.temperature);  // log2(e)/T
  a.c = float(C);
  a.Chi = float(C);
  a.Clo = float(C - double(a.Chi));
  const int maxslice = (a.nvec + a.S - 1) / a.S;
  const int run = maxslice / kCons + 2;  // running-sum length per thread per row slice
  a.bd.ex2 = float(kEx2RelErrBound);
  a.bd.gamma1 = float((3.0 + run) * 5.9604644775390625e-8 * 1.01);
  a.bd.xbar = float(std::log2(double(s.V)) + 2.0);
  a.out_tokens = s.out_tokens;
  a.out_n = s.out_n;
  a.err = s.err;
  a.row_info = s.row_info;
  a.q_at_d = s.q_at_d;
  a.p_at_d = s.p_at_d;
  cudaStream_t st = static_cast<cudaStream_t>(s.stream);
  if (cudaMemsetAsync(s.workspace, 0, wl.zero_bytes, st) != cudaSuccess) return SPEC_ECUDA;
  const size_t smem = sample_smem_bytes(2 * s.K + 1);
  if (s.dtype == SPEC_BF16) return launch_dataflow(verify_sample_kernel<EBf16>, a, smem, st);
  return launch_dataflow(verify_sample_kernel<EF32>, a, smem, st);
}

}  // namespace sv
