// Verification kernels: sampling mode (accept/reject + residual or bonus draw)
// and greedy mode (argmax match).
//
// Method ("aiengineeringfromscratch.com - Speculative decoding and EAGLE-3",
// "Variant: Leviathan rejection sampling", Steps 1-3; "devpost.com - phoenix",
// "What it does"): draft token d_i is accepted with probability
// min(1, q_i(d_i)/p_i(d_i)); at the first rejection j the correction is drawn
// from (q_j - p_j)+ normalised; after K acceptances a bonus token is drawn from
// q_K. Greedy mode accepts while d_i equals the target argmax.
//
// GB300 mapping. One thread-block cluster verifies one batch row. The C CTAs
// of the cluster split the vocabulary into C contiguous slices; every CTA
// streams its slice of all 2K logit rows (target and draft, positions
// 0..K-1) from HBM through a 4-stage shared-memory ring filled by 1-D bulk
// async copies (one producer thread, completion on mbarriers), while 8
// consumer warps compute per-row running maxima and sums of exp2. Per-CTA
// partials are exchanged through distributed shared memory, so every CTA holds
// the full softmax statistics of every row; the accept tests, the warp-ballot
// first-rejection search and the final draw are then computed without any
// global-memory scratch. The final draw re-reads only row j (target and
// draft, or target row K) while it is still resident in L2.
//
// Exactness. The fast path computes in fp32 with the MUFU exp2 and carries a
// proven bound on its error. A decision (accept test, or the inverse-CDF
// boundary of the drawn token) is taken from the fast path only when the
// uniform is farther from the decision threshold than twice that bound;
// otherwise the row is recomputed in double-float arithmetic (df.cuh), whose
// bound is ~1e-12, and flagged in row_info. This makes the output identical to
// an exact-arithmetic evaluation except in the (vanishing) cases flagged
// SPEC_ROW_UNCERTIFIED.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>

#include "../../include/specverify.h"
#include "common.cuh"
#include "df.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace sv {

// ============================================================== shared layout
struct Misc {
  int tok[kMaxK];
  float zt_d[kMaxK];  // target logit at the draft token, per position
  float zd_d[kMaxK];  // draft logit at the draft token
  float u[kMaxK + 1];
  int bad_token;
  int abort;
  int acc_state[kMaxK];
  double lq[kMaxK], lp[kMaxK];
  // exchange areas written by other CTAs of the cluster (DSMEM)
  double xR[kMaxCluster];
  float xQ[kMaxCluster], xP[kMaxCluster], xAq[kMaxCluster], xAp[kMaxCluster];
  double xS2[kMaxCluster][2];
  int dec_token;
  int dec_certified;
  // CTA-local
  double wR[kCW];
  float wQ[kCW], wP[kCW], wAq[kCW], wAp[kCW];
  double wS2[kCW][2];
  double accS[2];
  int best_idx[kMaxK + 1];  // greedy: combined argmax per row
};

struct Layout {
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  float* wM;      // [R][kCW]
  double* wS;     // [R][kCW]
  int* wI;        // [R][kCW]  (bad flag, or greedy index)
  float* cM;      // [kMaxCluster][R]
  double* cS;     // [kMaxCluster][R]
  int* cI;        // [kMaxCluster][R]
  float* rowM;    // [R]
  float* rowKc;   // [R]
  double* rowS;   // [R]
  double* rowN;   // [R]  log2 normaliser: Kc + log2(S)
  int* rowOK;     // [R]
  float* tab_hi;  // [256]
  float* tab_lo;  // [256]
  Misc* misc;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte size of the dynamic shared memory for R rows.
__host__ __device__ inline size_t smem_bytes(int R) {
  size_t o = 0;
  o += size_t(kStages) * kChunk;                 // ring
  o = align_up(o, 8) + 2 * kStages * 8;          // barriers
  o = align_up(o, 8) + size_t(R) * kCW * 8;      // wS
  o = align_up(o, 8) + size_t(kMaxCluster) * R * 8;  // cS
  o = align_up(o, 8) + size_t(R) * 8 * 2;        // rowS, rowN
  o = align_up(o, 8) + sizeof(Misc);
  o = align_up(o, 4) + size_t(R) * kCW * 4 * 2;  // wM, wI
  o += size_t(kMaxCluster) * R * 4 * 2;          // cM, cI
  o += size_t(R) * 4 * 3;                        // rowM, rowKc, rowOK
  o += 256 * 4 * 2;                              // table
  return align_up(o, 128);
}

__device__ inline Layout make_layout(uint8_t* base, int R) {
  Layout L;
  size_t o = 0;
  L.ring = base;
  o += size_t(kStages) * kChunk;
  o = align_up(o, 8);
  L.full = reinterpret_cast<uint64_t*>(base + o);
  L.empty = L.full + kStages;
  o += 2 * kStages * 8;
  o = align_up(o, 8);
  L.wS = reinterpret_cast<double*>(base + o);
  o += size_t(R) * kCW * 8;
  o = align_up(o, 8);
  L.cS = reinterpret_cast<double*>(base + o);
  o += size_t(kMaxCluster) * R * 8;
  o = align_up(o, 8);
  L.rowS = reinterpret_cast<double*>(base + o);
  L.rowN = L.rowS + R;
  o += size_t(R) * 8 * 2;
  o = align_up(o, 8);
  L.misc = reinterpret_cast<Misc*>(base + o);
  o += sizeof(Misc);
  o = align_up(o, 4);
  L.wM = reinterpret_cast<float*>(base + o);
  o += size_t(R) * kCW * 4;
  L.wI = reinterpret_cast<int*>(base + o);
  o += size_t(R) * kCW * 4;
  L.cM = reinterpret_cast<float*>(base + o);
  o += size_t(kMaxCluster) * R * 4;
  L.cI = reinterpret_cast<int*>(base + o);
  o += size_t(kMaxCluster) * R * 4;
  L.rowM = reinterpret_cast<float*>(base + o);
  L.rowKc = L.rowM + R;
  L.rowOK = reinterpret_cast<int*>(L.rowKc + R);
  o += size_t(R) * 4 * 3;
  L.tab_hi = reinterpret_cast<float*>(base + o);
  L.tab_lo = L.tab_hi + 256;
  return L;
}

// ============================================================== streaming
// Streams `nrows` row slices (vectors [vbeg, vend) of 16 bytes each) through
// the ring. Thread kCons issues the bulk copies; the kCons consumer threads
// call op.vec(vector, vector_index) for every vector and op.end_row(r) after
// each row. `it0` is the running chunk counter (ring phase); returns the new one.
template <class Op, class RowPtr>
__device__ uint32_t stream_rows(const Layout& L, uint32_t it0, int nrows, RowPtr rowptr, int vbeg,
                                int vend, Op& op, int32_t* err) {
  const int tid = threadIdx.x;
  const int nv = vend - vbeg;
  if (nv <= 0 || nrows <= 0) {
    if (tid < kCons) {
      for (int r = 0; r < nrows; ++r) {
        op.begin_row(r);
        op.end_row(r);
      }
    }
    return it0;
  }
  const int nchunk = (nv * 16 + kChunk - 1) / kChunk;
  const int cv = (nv + nchunk - 1) / nchunk;
  const uint32_t total = uint32_t(nrows) * nchunk;
  volatile int* abort_flag = &L.misc->abort;
  if (tid >= kCons) {
    if (tid == kCons) {
      for (uint32_t q = 0; q < total; ++q) {
        const uint32_t it = it0 + q;
        const int stage = it % kStages;
        if (it >= kStages) {
          if (*abort_flag || !mbar_wait(&L.empty[stage], ((it / kStages) - 1) & 1)) {
            *abort_flag = 1;
            break;
          }
        }
        const int r = q / nchunk, k = q % nchunk;
        const int c0 = vbeg + k * cv;
        const int c1 = min(vend, c0 + cv);
        const uint32_t bytes = uint32_t(c1 - c0) * 16u;
        const char* src = reinterpret_cast<const char*>(rowptr(r)) + size_t(c0) * 16;
        mbar_arrive_expect_tx(&L.full[stage], bytes);
        bulk_g2s(L.ring + size_t(stage) * kChunk, src, bytes, &L.full[stage]);
      }
    }
  } else {
    const int lane = tid & 31;
    for (int r = 0; r < nrows; ++r) {
      op.begin_row(r);
      for (int k = 0; k < nchunk; ++k) {
        const uint32_t it = it0 + uint32_t(r) * nchunk + k;
        const int stage = it % kStages;
        bool ok = !*abort_flag && mbar_wait(&L.full[stage], (it / kStages) & 1);
        if (!ok) {
          *abort_flag = 1;
          continue;
        }
        const int c0 = vbeg + k * cv;
        const int c1 = min(vend, c0 + cv);
        const uint4* buf = reinterpret_cast<const uint4*>(L.ring + size_t(stage) * kChunk);
        for (int i = tid; i < c1 - c0; i += kCons) op.vec(buf[i], c0 + i);
        __syncwarp();
        if (lane == 0) mbar_arrive(&L.empty[stage]);
      }
      op.end_row(r);
    }
  }
  if (tid == 0 && *abort_flag && err) atomicOr(err, SPEC_DERR_TIMEOUT);
  return it0 + total;
}

// ============================================================== softmax stats
// Running (max, sum of exp2(z*c - Kc)) of one row slice per thread. Kc is an
// integer offset derived from the running max; when the max grows the sum is
// rescaled by an exact power of two.
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
    double s = 0.0;
    if (S != 0.0f) {
      const float Kw = offset_of(Mw, c);
      s = ldexp(static_cast<double>(S), static_cast<int>(Kc - Kw));
    }
    s = warp_sum_d(s);
    const int anybad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      const int rr = row_base + r;
      L->wM[rr * kCW + warp] = Mw;
      L->wS[rr * kCW + warp] = s;
      L->wI[rr * kCW + warp] = anybad;
    }
  }
};

// Combines the per-warp partials of rows [r0, r1) into one partial per CTA and
// stores it into slot [crank][r] of every CTA of the cluster.
__device__ void stats_cta_broadcast(const Layout& L, int R, int r0, int r1, float c, int crank,
                                    int csize) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kCW) return;
  for (int r = r0 + warp; r < r1; r += kCW) {
    const float m = lane < kCW ? L.wM[r * kCW + lane] : -INFINITY;
    const double sw = lane < kCW ? L.wS[r * kCW + lane] : 0.0;
    const int bw = lane < kCW ? L.wI[r * kCW + lane] : 0;
    const float Mc = warp_max_f(m);
    double s = 0.0;
    if (sw != 0.0) s = ldexp(sw, static_cast<int>(offset_of(m, c) - offset_of(Mc, c)));
    s = warp_sum_d(s);
    const int bad = __any_sync(0xffffffffu, bw);
    if (lane < csize) {
      const uint32_t q = lane;
      st_cluster_f32(mapa_shared(smem_u32(&L.cM[crank * R + r]), q), Mc);
      st_cluster_f64(mapa_shared(smem_u32(&L.cS[crank * R + r]), q), s);
      st_cluster_u32(mapa_shared(smem_u32(&L.cI[crank * R + r]), q), uint32_t(bad));
    }
  }
}

// Final statistics of rows [r0, r1) from the C gathered partials (identical in
// every CTA: same values, same order).
__device__ void stats_final(const Layout& L, int R, int r0, int r1, float c, int csize) {
  for (int r = r0 + int(threadIdx.x); r < r1; r += blockDim.x) {
    float M = -INFINITY;
    int bad = 0;
    for (int q = 0; q < csize; ++q) {
      M = fmaxf(M, L.cM[q * R + r]);
      bad |= L.cI[q * R + r];
    }
    const float Kc = offset_of(M, c);
    double S = 0.0;
    for (int q = 0; q < csize; ++q) {
      const double sq = L.cS[q * R + r];
      if (sq != 0.0) S += ldexp(sq, static_cast<int>(offset_of(L.cM[q * R + r], c) - Kc));
    }
    const bool ok = !bad && isfinite(M) && fabsf(Kc) < 4194304.0f && S > 0.0 && isfinite(S);
    L.rowM[r] = M;
    L.rowKc[r] = Kc;
    L.rowS[r] = S;
    L.rowN[r] = ok ? static_cast<double>(Kc) + log2(S) : 0.0;
    L.rowOK[r] = ok ? 1 : 0;
  }
}

// ============================================================== error model
// Bound on the relative error of ex2.approx.ftz.f32 over [-126, 1], measured
// exhaustively on GB300 (every fp32 input in the range against an fp64
// reference); passed in by the host.
struct Bounds {
  double ex2;     // ex2.approx relative error bound
  double gamma1;  // relative error bound of the pass-1 fp32 summation
  double xbar;    // bound on sum_v q_v |x_v| used before pass 2 (entropy bound)
};

// log2-domain error bound of log2 q(d) from the fast statistics:
// |err| <= (delta_S / ln2 + u (|x_d| + xbar + 2)) * 1.02,
// delta_S = ex2 + ln2 u xbar + gamma1 (relative error of the row sum).
__device__ inline double log2_prob_bound(const Bounds& bd, double x_d) {
  const double dS = bd.ex2 + kLn2 * kUd * bd.xbar + bd.gamma1;
  return (dS / kLn2 + kUd * (fabs(x_d) + bd.xbar + 2.0)) * 1.02;
}

// ============================================================== accurate path
__device__ __forceinline__ df acc_elem(float z, float Chi, float Clo, float Ohi, float Olo,
                                       const float* th, const float* tl) {
  const df p = two_prod(z, Chi);
  const float pl = __fmaf_rn(z, Clo, p.lo);
  const df s = two_sum(p.hi, -Ohi);
  const float xl = __fadd_rn(s.lo, __fsub_rn(pl, Olo));
  return df_exp2(s.hi, xl, th, tl);
}

// Relative error bound of one acc_elem value including its normaliser.
constexpr double kAccRho = 4e-12;

__device__ inline void load_table(const Layout& L) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    L.tab_hi[i] = kExp2Tab.hi[i];
    L.tab_lo[i] = kExp2Tab.lo[i];
  }
}

// Block sum of a per-thread double (consumer warps only contribute) -> returned in all threads.
__device__ double block_sum_consumers(const Layout& L, double v, int slot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_sum_d(v);
  if (warp < kCW && lane == 0) L.misc->wS2[warp][slot] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < kCW; ++w) t += L.misc->wS2[w][slot];
  __syncthreads();
  return t;
}

// Accurate sum_v 2^(z_v C - Kc) over the cluster, for up to two rows at once.
// Every CTA returns the same values.
template <class E>
__device__ void acc_norms(const Layout& L, const typename E::T* row0, float Kc0,
                          const typename E::T* row1, float Kc1, int vbeg, int vend, float Chi,
                          float Clo, int crank, int csize, double* out) {
  const int tid = threadIdx.x;
  df a0{0.f, 0.f}, a1{0.f, 0.f};
  if (tid < kCons) {
    const uint4* p0 = reinterpret_cast<const uint4*>(row0);
    const uint4* p1 = row1 ? reinterpret_cast<const uint4*>(row1) : nullptr;
    for (int vi = vbeg + tid; vi < vend; vi += kCons) {
      float z[E::kVec];
      E::unpack(ldg_nc_v4(p0 + vi), z);
#pragma unroll
      for (int k = 0; k < E::kVec; ++k)
        a0 = df_add(a0, acc_elem(z[k], Chi, Clo, Kc0, 0.f, L.tab_hi, L.tab_lo));
      if (p1) {
        E::unpack(ldg_nc_v4(p1 + vi), z);
#pragma unroll
        for (int k = 0; k < E::kVec; ++k)
          a1 = df_add(a1, acc_elem(z[k], Chi, Clo, Kc1, 0.f, L.tab_hi, L.tab_lo));
      }
    }
  }
  const double s0 = block_sum_consumers(L, df_to_double(a0), 0);
  const double s1 = block_sum_consumers(L, df_to_double(a1), 1);
  if (threadIdx.x < csize) {
    const uint32_t q = threadIdx.x;
    st_cluster_f64(mapa_shared(smem_u32(&L.misc->xS2[crank][0]), q), s0);
    st_cluster_f64(mapa_shared(smem_u32(&L.misc->xS2[crank][1]), q), s1);
  }
  cluster_sync();
  double t0 = 0.0, t1 = 0.0;
  for (int q = 0; q < csize; ++q) {
    t0 += L.misc->xS2[q][0];
    t1 += L.misc->xS2[q][1];
  }
  out[0] = t0;
  out[1] = t1;
  cluster_sync();  // the exchange slots may be reused after this point
}

// ============================================================== final draw
// Per-vector residual entries of the fast path (fp32, MUFU exp2).
template <class E>
struct FastResidual {
  const uint4* tq;  // target row j (or K), as 16-byte vectors
  const uint4* tp;  // draft row j, or null for a draw from q alone
  float c;
  float Oq, Fq, Op, Fp;
  // r[k] entries and their pairwise fp32 sum (the value scanned at vector level).
  __device__ __forceinline__ float entries(int vi, float (&r)[E::kVec], float& q_sum,
                                           float& p_sum, float& aq, float& ap) const {
    float zq[E::kVec];
    E::unpack(ldg_nc_v4(tq + vi), zq);
    float zp[E::kVec];
    if (tp) E::unpack(ldg_nc_v4(tp + vi), zp);
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      const float xa = __fmaf_rn(zq[k], c, -Oq);
      const float q = __fmul_rn(ex2_approx(xa), Fq);
      q_sum = __fadd_rn(q_sum, q);
      aq = __fmaf_rn(q, fminf(-xa, 1.0e4f), aq);
      if (tp) {
        const float xb = __fmaf_rn(zp[k], c, -Op);
        const float p = __fmul_rn(ex2_approx(xb), Fp);
        p_sum = __fadd_rn(p_sum, p);
        ap = __fmaf_rn(p, fminf(-xb, 1.0e4f), ap);
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
};

// Per-vector residual entries of the accurate path (double-float).
template <class E>
struct AccResidual {
  const uint4* tq;
  const uint4* tp;
  float Chi, Clo;
  float Oq_hi, Oq_lo, Op_hi, Op_lo;
  const float* th;
  const float* tl;
  __device__ __forceinline__ double entries(int vi, double (&r)[E::kVec], double& q_sum,
                                            double& p_sum) const {
    float zq[E::kVec];
    E::unpack(ldg_nc_v4(tq + vi), zq);
    float zp[E::kVec];
    if (tp) E::unpack(ldg_nc_v4(tp + vi), zp);
    double vs = 0.0;
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      const df q = acc_elem(zq[k], Chi, Clo, Oq_hi, Oq_lo, th, tl);
      q_sum += df_to_double(q);
      df rk = q;
      if (tp) {
        const df p = acc_elem(zp[k], Chi, Clo, Op_hi, Op_lo, th, tl);
        p_sum += df_to_double(p);
        rk = df_sub(q, p);
      }
      double rv = df_to_double(rk);
      if (!(rv > 0.0)) rv = 0.0;
      r[k] = rv;
      vs += rv;
    }
    return vs;
  }
};

// Warp w's contiguous range of the CTA's vector slice [vbeg, vend).
__device__ __forceinline__ void warp_range(int vbeg, int vend, int w, int& wb, int& we) {
  const long n = vend - vbeg;
  wb = vbeg + int(n * w / kCW);
  we = vbeg + int(n * (w + 1) / kCW);
}

struct Draw {
  int token;      // drawn vocabulary index (-1: none found)
  double lo, hi;  // computed cumulative mass before / through the drawn token
};

// Fine search inside one warp range for the first entry whose cumulative mass
// exceeds t. `base` is the computed mass before the range. Lanes scan vectors
// in the same order as the sweep: iteration-major, lane-minor.
template <int kVec, class EntriesFn>
__device__ Draw warp_search(int wb, int we, double base, double t, EntriesFn entries) {
  const int lane = threadIdx.x & 31;
  Draw d{-1, base, base};
  int last_pos = -1;
  double last_lo = base, last_hi = base;
  for (int v0 = wb; v0 < we; v0 += 32) {
    const int vi = v0 + lane;
    double r[kVec];
    double vs = 0.0;
    if (vi < we) vs = entries(vi, r);
    else
      for (int k = 0; k < kVec; ++k) r[k] = 0.0;
    // inclusive scan of vector sums across lanes
    double inc = vs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const double tot = __shfl_sync(0xffffffffu, inc, 31);
    const unsigned hit = __ballot_sync(0xffffffffu, base + inc > t);
    if (hit) {
      const int l = __ffs(hit) - 1;
      int tok = -1;
      double lo = 0.0, hi = 0.0;
      int lp = -1;
      double llo = 0.0, lhi = 0.0;
      if (lane == l) {
        double c0 = base + (inc - vs);
        for (int k = 0; k < kVec; ++k) {
          const double c1 = c0 + r[k];
          if (r[k] > 0.0) {
            lp = vi * kVec + k;
            llo = c0;
            lhi = c1;
          }
          if (c1 > t && tok < 0 && r[k] > 0.0) {
            tok = vi * kVec + k;
            lo = c0;
            hi = c1;
          }
          c0 = c1;
        }
        if (tok < 0) {  // rounding of the vector sum: take the last positive entry
          tok = lp;
          lo = llo;
          hi = lhi;
        }
      }
      d.token = __shfl_sync(0xffffffffu, tok, l);
      d.lo = __shfl_sync(0xffffffffu, lo, l);
      d.hi = __shfl_sync(0xffffffffu, hi, l);
      if (d.token >= 0) return d;
    }
    // remember the last positive entry of this iteration (fallback when t is past the end)
    int lp = -1;
    double llo = 0.0, lhi = 0.0;
    double c0 = base + (inc - vs);
    for (int k = 0; k < kVec; ++k) {
      const double c1 = c0 + r[k];
      if (r[k] > 0.0 && vi < we) {
        lp = vi * kVec + k;
        llo = c0;
        lhi = c1;
      }
      c0 = c1;
    }
    const unsigned has = __ballot_sync(0xffffffffu, lp >= 0);
    if (has) {
      const int l = 31 - __clz(has);
      last_pos = __shfl_sync(0xffffffffu, lp, l);
      last_lo = __shfl_sync(0xffffffffu, llo, l);
      last_hi = __shfl_sync(0xffffffffu, lhi, l);
    }
    base += tot;
  }
  d.token = last_pos;
  d.lo = last_lo;
  d.hi = last_hi;
  return d;
}

// ============================================================== sampling kernel
struct VerifyArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  int B, K, V;
  float c;         // fl32(log2(e) / T)
  float Chi, Clo;  // log2(e) / T as a float pair
  double C;        // log2(e) / T in fp64
  Bounds bd;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  int32_t* row_info;
  float* q_at_d;
  float* p_at_d;
};

enum { kAccept = 0, kReject = 1, kAmbiguous = 2, kInvalid = 3 };

template <class E>
__global__ void __launch_bounds__(kThreads, 1) verify_sample_kernel(const VerifyArgs a) {
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K, V = a.V, R = 2 * K + 1;
  const Layout L = make_layout(smem_raw, R);
  Misc& ms = *L.misc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int crank = int(cluster_ctarank()), csize = int(cluster_nctarank());
  const int b = blockIdx.x / csize;
  const T* tgt = static_cast<const T*>(a.target) + size_t(b) * (K + 1) * V;
  const T* drf = static_cast<const T*>(a.draft) + size_t(b) * K * V;
  const int nvec = V / E::kVec;
  const int vbeg = int(int64_t(nvec) * crank / csize);
  const int vend = int(int64_t(nvec) * (crank + 1) / csize);
  const float c = a.c;

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&L.full[s], 1);
      mbar_init(&L.empty[s], kCW);
    }
    ms.abort = 0;
    ms.bad_token = 0;
    fence_mbar_init();
  }
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
  __syncthreads();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // ---------------------------------------------------------------- pass 1
  StatOp<E> op;
  op.c = c;
  op.row_base = 0;
  op.L = &L;
  auto rp1 = [&](int r) -> const T* {
    const int i = r >> 1;
    return (r & 1) ? drf + size_t(i) * V : tgt + size_t(i) * V;
  };
  uint32_t it = stream_rows(L, 0u, 2 * K, rp1, vbeg, vend, op, a.err);
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  stats_cta_broadcast(L, R, 0, 2 * K, c, crank, csize);
  cluster_sync();
  stats_final(L, R, 0, 2 * K, c, csize);
  __syncthreads();

  // ---------------------------------------------------------------- accept tests
  // Every CTA evaluates the same tests on the same gathered statistics.
  if (warp == 0 && lane < K) {
    const int i = lane;
    const int rt = 2 * i, rd = 2 * i + 1;
    int st;
    double lq = 0.0, lp = 0.0;
    if (ms.bad_token || !L.rowOK[rt] || !L.rowOK[rd]) {
      st = kInvalid;
    } else {
      const float zt = ms.zt_d[i], zd = ms.zd_d[i];
      // log2 q(d) = z c - (Kc + log2 S) in the fp32-temperature scale
      lq = double(zt) * double(c) - L.rowN[rt];
      lp = double(zd) * double(c) - L.rowN[rd];
      const double u = ms.u[i];
      if (zd == -INFINITY) {
        st = kAccept;  // p(d) = 0 accepts
      } else if (zt == -INFINITY) {
        st = kReject;  // q(d) = 0 < u is impossible, u < 0 never holds
      } else {
        const double xt = double(zt) * double(c) - double(L.rowKc[rt]);
        const double xd = double(zd) * double(c) - double(L.rowKc[rd]);
        const double beta = kLn2 * (log2_prob_bound(a.bd, xt) + log2_prob_bound(a.bd, xd)) * 1.02;
        const double ratio = exp2(lq - lp);
        const double rlo = fmin(1.0, ratio * (1.0 - beta));
        const double rhi = fmin(1.0, ratio * (1.0 + beta));
        st = (u < rlo) ? kAccept : (u >= rhi ? kReject : kAmbiguous);
      }
    }
    ms.acc_state[i] = st;
    ms.lq[i] = lq;
    ms.lp[i] = lp;
  }
  __syncthreads();

  int flags = 0;
  int n = 0;
  bool error = ms.bad_token != 0;
  for (;;) {
    int i = n;
    while (i < K && ms.acc_state[i] == kAccept) ++i;
    if (i == K) {
      n = K;
      break;
    }
    const int st = ms.acc_state[i];
    if (st == kInvalid) {
      error = true;
      n = i;
      break;
    }
    if (st == kReject) {
      n = i;
      break;
    }
    // ambiguous: decide with accurate normalisers of rows 2i and 2i+1
    flags |= SPEC_ROW_ACCEPT_REFINED;
    load_table(L);
    __syncthreads();
    double S2[2];
    acc_norms<E>(L, tgt + size_t(i) * V, L.rowKc[2 * i], drf + size_t(i) * V, L.rowKc[2 * i + 1],
                 vbeg, vend, a.Chi, a.Clo, crank, csize, S2);
    const double lqa = double(ms.zt_d[i]) * a.C - double(L.rowKc[2 * i]) - log2(S2[0]);
    const double lpa = double(ms.zd_d[i]) * a.C - double(L.rowKc[2 * i + 1]) - log2(S2[1]);
    const double ratio = fmin(1.0, exp2(lqa - lpa));
    const double u = ms.u[i];
    if (fabs(u - ratio) <= 1e-10 * ratio) flags |= SPEC_ROW_UNCERTIFIED;
    __syncthreads();
    if (u < ratio) {
      if (tid == 0) ms.acc_state[i] = kAccept;
      __syncthreads();
      n = i + 1;
      continue;
    }
    n = i;
    break;
  }

  // ---------------------------------------------------------------- final draw
  int token = -1;
  if (!error) {
    const bool bonus = (n == K);
    int rq, rpd;
    if (bonus) {
      rq = 2 * K;
      rpd = -1;
      // statistics of target row K (streamed from HBM through the ring)
      StatOp<E> opk;
      opk.c = c;
      opk.row_base = 2 * K;
      opk.L = &L;
      auto rpk = [&](int) -> const T* { return tgt + size_t(K) * V; };
      it = stream_rows(L, it, 1, rpk, vbeg, vend, opk, a.err);
      __syncthreads();
      stats_cta_broadcast(L, R, 2 * K, 2 * K + 1, c, crank, csize);
      cluster_sync();
      stats_final(L, R, 2 * K, 2 * K + 1, c, csize);
      __syncthreads();
      if (!L.rowOK[2 * K]) error = true;
    } else {
      rq = 2 * n;
      rpd = 2 * n + 1;
    }
    if (!error) {
      const int jrow = bonus ? K : n;
      const uint4* vq = reinterpret_cast<const uint4*>(tgt + size_t(jrow) * V);
      const uint4* vp = bonus ? nullptr : reinterpret_cast<const uint4*>(drf + size_t(n) * V);
      const double u = ms.u[K];
      // ---------------- fast sweep
      FastResidual<E> fr;
      fr.tq = vq;
      fr.tp = vp;
      fr.c = c;
      {
        const double Nq = L.rowN[rq];
        fr.Oq = float(Nq);
        fr.Fq = float(exp2(-(Nq - double(fr.Oq))));
        if (!bonus) {
          const double Np = L.rowN[rpd];
          fr.Op = float(Np);
          fr.Fp = float(exp2(-(Np - double(fr.Op))));
        } else {
          fr.Op = 0.f;
          fr.Fp = 0.f;
        }
      }
      int wb, we;
      warp_range(vbeg, vend, warp < kCW ? warp : 0, wb, we);
      {
        double R_ = 0.0;
        float Q = 0.f, P = 0.f, Aq = 0.f, Ap = 0.f;
        if (warp < kCW) {
          for (int vi = wb + lane; vi < we; vi += 32) {
            float r[E::kVec];
            const float vs = fr.entries(vi, r, Q, P, Aq, Ap);
            R_ += double(vs);
          }
          R_ = warp_sum_d(R_);
          Q = warp_sum_f(Q);
          P = warp_sum_f(P);
          Aq = warp_sum_f(Aq);
          Ap = warp_sum_f(Ap);
          if (lane == 0) {
            ms.wR[warp] = R_;
            ms.wQ[warp] = Q;
            ms.wP[warp] = P;
            ms.wAq[warp] = Aq;
            ms.wAp[warp] = Ap;
          }
        }
      }
      __syncthreads();
      if (tid < csize) {
        double Rc = 0.0;
        float Qc = 0.f, Pc = 0.f, Aqc = 0.f, Apc = 0.f;
        for (int w = 0; w < kCW; ++w) {
          Rc += ms.wR[w];
          Qc += ms.wQ[w];
          Pc += ms.wP[w];
          Aqc += ms.wAq[w];
          Apc += ms.wAp[w];
        }
        const uint32_t q = tid;
        st_cluster_f64(mapa_shared(smem_u32(&ms.xR[crank]), q), Rc);
        st_cluster_f32(mapa_shared(smem_u32(&ms.xQ[crank]), q), Qc);
        st_cluster_f32(mapa_shared(smem_u32(&ms.xP[crank]), q), Pc);
        st_cluster_f32(mapa_shared(smem_u32(&ms.xAq[crank]), q), Aqc);
        st_cluster_f32(mapa_shared(smem_u32(&ms.xAp[crank]), q), Apc);
      }
      cluster_sync();
      double Sr = 0.0, Qt = 0.0, Pt = 0.0, Aqt = 0.0, Apt = 0.0;
      for (int q = 0; q < csize; ++q) {
        Sr += ms.xR[q];
        Qt += ms.xQ[q];
        Pt += ms.xP[q];
        Aqt += ms.xAq[q];
        Apt += ms.xAp[q];
      }
      // error bound of the fast sweep (absolute, in probability units)
      double E_;
      {
        const double u32 = kUd;
        auto side = [&](double Qs, double A, int row) {
          const double l2S = fabs(log2(L.rowS[row]));
          const double xb = A / fmax(Qs, 1e-300) + l2S + 1.0;
          const double rho = 2.0 * a.bd.ex2 + 2.0 * u32 + a.bd.gamma1 +
                             kLn2 * u32 * (2.0 * A / fmax(Qs, 1e-300) + 2.0 * xb + l2S + 2.0);
          return 1.02 * fmax(Qs, 1.0) * rho;
        };
        E_ = side(Qt, Aqt, rq) + (bonus ? 0.0 : side(Pt, Apt, rpd)) + 8.0 * u32 * Sr + 1e-30;
      }
      const double tstar = u * Sr;
      bool certified = false;
      if (Sr > 2.0 * E_) {
        // locate the CTA, then the warp, holding t*
        int cs = -1;
        double pre = 0.0, pre_cs = 0.0;
        for (int q = 0; q < csize; ++q) {
          if (ms.xR[q] > 0.0) {
            cs = q;
            pre_cs = pre;
          }
          if (pre + ms.xR[q] > tstar && ms.xR[q] > 0.0) {
            cs = q;
            pre_cs = pre;
            break;
          }
          pre += ms.xR[q];
        }
        if (crank == cs) {
          int ws = -1;
          double wpre = pre_cs, wpre_s = pre_cs;
          for (int w = 0; w < kCW; ++w) {
            if (ms.wR[w] > 0.0) {
              ws = w;
              wpre_s = wpre;
            }
            if (wpre + ms.wR[w] > tstar && ms.wR[w] > 0.0) {
              ws = w;
              wpre_s = wpre;
              break;
            }
            wpre += ms.wR[w];
          }
          if (warp == ws) {
            int swb, swe;
            warp_range(vbeg, vend, ws, swb, swe);
            auto ent = [&](int vi, double (&rd)[E::kVec]) -> double {
              float r[E::kVec];
              float q0 = 0.f, p0 = 0.f, a0 = 0.f, a1 = 0.f;
              const float vs = fr.entries(vi, r, q0, p0, a0, a1);
#pragma unroll
              for (int k = 0; k < E::kVec; ++k) rd[k] = double(r[k]);
              return double(vs);
            };
            const Draw d = warp_search<E::kVec>(swb, swe, wpre_s, tstar, ent);
            if (lane == 0) {
              const double margin = fmin(tstar - d.lo, d.hi - tstar);
              const int cert = (d.token >= 0 && margin > 2.0 * E_ + 4e-16 * Sr) ? 1 : 0;
              for (int q = 0; q < csize; ++q) {
                st_cluster_u32(mapa_shared(smem_u32(&ms.dec_token), q), uint32_t(d.token));
                st_cluster_u32(mapa_shared(smem_u32(&ms.dec_certified), q), uint32_t(cert));
              }
            }
          }
        }
        cluster_sync();
        certified = ms.dec_certified != 0;
        token = ms.dec_token;
      }
      if (!certified) {
        // ---------------- accurate fallback (double-float)
        flags |= SPEC_ROW_SAMPLE_REFINED;
        load_table(L);
        __syncthreads();
        double S2[2];
        acc_norms<E>(L, tgt + size_t(jrow) * V, L.rowKc[rq], bonus ? nullptr : drf + size_t(n) * V,
                     bonus ? 0.f : L.rowKc[rpd], vbeg, vend, a.Chi, a.Clo, crank, csize, S2);
        AccResidual<E> ar;
        ar.tq = vq;
        ar.tp = vp;
        ar.Chi = a.Chi;
        ar.Clo = a.Clo;
        ar.th = L.tab_hi;
        ar.tl = L.tab_lo;
        {
          const double Oq = double(L.rowKc[rq]) + log2(S2[0]);
          ar.Oq_hi = float(Oq);
          ar.Oq_lo = float(Oq - double(ar.Oq_hi));
          if (!bonus) {
            const double Op = double(L.rowKc[rpd]) + log2(S2[1]);
            ar.Op_hi = float(Op);
            ar.Op_lo = float(Op - double(ar.Op_hi));
          }
        }
        for (int pass = 0; pass < 2; ++pass) {
          double R2 = 0.0, Q2 = 0.0, P2 = 0.0;
          if (warp < kCW) {
            for (int vi = wb + lane; vi < we; vi += 32) {
              double r[E::kVec];
              R2 += ar.entries(vi, r, Q2, P2);
            }
            R2 = warp_sum_d(R2);
            Q2 = warp_sum_d(Q2);
            P2 = warp_sum_d(P2);
            if (lane == 0) {
              ms.wR[warp] = R2;
              ms.wS2[warp][0] = Q2;
              ms.wS2[warp][1] = P2;
            }
          }
          __syncthreads();
          if (tid < csize) {
            double Rc = 0.0, Qc = 0.0, Pc = 0.0;
            for (int w = 0; w < kCW; ++w) {
              Rc += ms.wR[w];
              Qc += ms.wS2[w][0];
              Pc += ms.wS2[w][1];
            }
            const uint32_t q = tid;
            st_cluster_f64(mapa_shared(smem_u32(&ms.xR[crank]), q), Rc);
            st_cluster_f64(mapa_shared(smem_u32(&ms.xS2[crank][0]), q), Qc);
            st_cluster_f64(mapa_shared(smem_u32(&ms.xS2[crank][1]), q), Pc);
          }
          cluster_sync();
          double Sr2 = 0.0, Qt2 = 0.0, Pt2 = 0.0;
          for (int q = 0; q < csize; ++q) {
            Sr2 += ms.xR[q];
            Qt2 += ms.xS2[q][0];
            Pt2 += ms.xS2[q][1];
          }
          if (Sr2 == 0.0 && ar.tp != nullptr) {
            // zero residual mass: the draw uses q_j itself
            flags |= SPEC_ROW_ZERO_RESIDUAL;
            ar.tp = nullptr;
            cluster_sync();
            continue;
          }
          const double E2 = kAccRho * (Qt2 + Pt2) + 1e-14 * Sr2 + 1e-300;
          const double t2 = u * Sr2;
          int cs = -1;
          double pre = 0.0, pre_cs = 0.0;
          for (int q = 0; q < csize; ++q) {
            if (ms.xR[q] > 0.0) {
              cs = q;
              pre_cs = pre;
            }
            if (pre + ms.xR[q] > t2 && ms.xR[q] > 0.0) {
              cs = q;
              pre_cs = pre;
              break;
            }
            pre += ms.xR[q];
          }
          if (crank == cs) {
            int ws = -1;
            double wpre = pre_cs, wpre_s = pre_cs;
            for (int w = 0; w < kCW; ++w) {
              if (ms.wR[w] > 0.0) {
                ws = w;
                wpre_s = wpre;
              }
              if (wpre + ms.wR[w] > t2 && ms.wR[w] > 0.0) {
                ws = w;
                wpre_s = wpre;
                break;
              }
              wpre += ms.wR[w];
            }
            if (warp == ws) {
              int swb, swe;
              warp_range(vbeg, vend, ws, swb, swe);
              auto ent = [&](int vi, double (&rd)[E::kVec]) -> double {
                double q0 = 0.0, p0 = 0.0;
                return ar.entries(vi, rd, q0, p0);
              };
              const Draw d = warp_search<E::kVec>(swb, swe, wpre_s, t2, ent);
              if (lane == 0) {
                const double margin = fmin(t2 - d.lo, d.hi - t2);
                const int cert = (d.token >= 0 && margin > 2.0 * E2) ? 1 : 0;
                for (int q = 0; q < csize; ++q) {
                  st_cluster_u32(mapa_shared(smem_u32(&ms.dec_token), q), uint32_t(d.token));
                  st_cluster_u32(mapa_shared(smem_u32(&ms.dec_certified), q), uint32_t(cert));
                }
              }
            }
          }
          cluster_sync();
          token = ms.dec_token;
          if (!ms.dec_certified) flags |= SPEC_ROW_UNCERTIFIED;
          break;
        }
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
        atomicOr(a.err, ms.bad_token ? SPEC_DERR_TOKEN : SPEC_DERR_LOGITS);
      }
    }
    if (warp == 0 && lane < K && a.q_at_d) {
      const int i = lane;
      const bool ok = !ms.bad_token && L.rowOK[2 * i] && L.rowOK[2 * i + 1];
      a.q_at_d[size_t(b) * K + i] = ok ? float(exp2(ms.lq[i])) : -1.0f;
      a.p_at_d[size_t(b) * K + i] = ok ? float(exp2(ms.lp[i])) : -1.0f;
    }
  }
  // no CTA leaves while another may still address its shared memory
  cluster_sync();
}

// ============================================================== greedy kernel
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
      if (ob > best || (ob == best && oi < idx)) {
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

__device__ void argmax_cta_broadcast(const Layout& L, int R, int r0, int r1, int crank, int csize) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kCW) return;
  for (int r = r0 + warp; r < r1; r += kCW) {
    float best = lane < kCW ? L.wM[r * kCW + lane] : -INFINITY;
    int idx = lane < kCW ? L.wI[r * kCW + lane] : INT_MAX;
    int bad = (idx == -2);
    if (bad) idx = INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ob > best || (ob == best && oi < idx)) {
        best = ob;
        idx = oi;
      }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane < csize) {
      const uint32_t q = lane;
      st_cluster_f32(mapa_shared(smem_u32(&L.cM[crank * R + r]), q), best);
      st_cluster_u32(mapa_shared(smem_u32(&L.cI[crank * R + r]), q), uint32_t(bad ? -2 : idx));
    }
  }
}

__device__ void argmax_final(const Layout& L, int R, int r0, int r1, int csize) {
  for (int r = r0 + int(threadIdx.x); r < r1; r += blockDim.x) {
    float best = -INFINITY;
    int idx = INT_MAX;
    int bad = 0;
    for (int q = 0; q < csize; ++q) {
      const float b = L.cM[q * R + r];
      const int i = L.cI[q * R + r];
      if (i == -2) {
        bad = 1;
        continue;
      }
      if (b > best || (b == best && i < idx)) {
        best = b;
        idx = i;
      }
    }
    L.misc->best_idx[r] = (bad || idx == INT_MAX) ? -1 : idx;
  }
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
__global__ void __launch_bounds__(kThreads, 1) verify_greedy_kernel(const GreedyArgs a) {
  using T = typename E::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K, V = a.V, R = K + 1;
  const Layout L = make_layout(smem_raw, R);
  Misc& ms = *L.misc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int crank = int(cluster_ctarank()), csize = int(cluster_nctarank());
  const int b = blockIdx.x / csize;
  const T* tgt = static_cast<const T*>(a.target) + size_t(b) * (K + 1) * V;
  const int nvec = V / E::kVec;
  const int vbeg = int(int64_t(nvec) * crank / csize);
  const int vend = int(int64_t(nvec) * (crank + 1) / csize);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&L.full[s], 1);
      mbar_init(&L.empty[s], kCW);
    }
    ms.abort = 0;
    fence_mbar_init();
  }
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
  __syncthreads();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  ArgmaxOp<E> op;
  op.row_base = 0;
  op.L = &L;
  auto rp = [&](int r) -> const T* { return tgt + size_t(r) * V; };
  uint32_t it = stream_rows(L, 0u, K, rp, vbeg, vend, op, a.err);
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  argmax_cta_broadcast(L, R, 0, K, crank, csize);
  cluster_sync();
  argmax_final(L, R, 0, K, csize);
  __syncthreads();

  // first mismatch by warp ballot
  bool error = ms.bad_token != 0;
  int n = K;
  {
    int bad_any = 0;
    unsigned mism = 0;
    if (warp == 0) {
      const int g = lane < K ? ms.best_idx[lane] : 0;
      const bool m = lane < K && g != ms.tok[lane];
      mism = __ballot_sync(0xffffffffu, m);
      bad_any = __any_sync(0xffffffffu, lane < K && g < 0);
    }
    if (tid == 0) {
      ms.acc_state[0] = mism ? (__ffs(mism) - 1) : K;
      ms.acc_state[1] = bad_any;
    }
    __syncthreads();
    n = ms.acc_state[0];
    // a NaN row matters only up to the first mismatch
    for (int i = 0; i <= min(n, K - 1); ++i)
      if (ms.best_idx[i] < 0) error = true;
  }
  int token = -1;
  if (!error) {
    if (n < K) {
      token = ms.best_idx[n];
    } else {
      op.row_base = K;
      auto rpk = [&](int) -> const T* { return tgt + size_t(K) * V; };
      it = stream_rows(L, it, 1, rpk, vbeg, vend, op, a.err);
      __syncthreads();
      argmax_cta_broadcast(L, R, K, K + 1, crank, csize);
      cluster_sync();
      argmax_final(L, R, K, K + 1, csize);
      __syncthreads();
      token = ms.best_idx[K];
      if (token < 0) error = true;
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
      if (error && a.err) atomicOr(a.err, ms.bad_token ? SPEC_DERR_TOKEN : SPEC_DERR_LOGITS);
    }
  }
  cluster_sync();
}

// ============================================================== host launch
namespace {

int pick_cluster(int B, int nvec) {
  int c = 16;
  if (const char* e = getenv("SPECVERIFY_CLUSTER")) c = atoi(e);
  else if (B >= 128) c = 8;
  if (c != 1 && c != 2 && c != 4 && c != 8 && c != 16) c = 8;
  while (c > 1 && c > nvec) c >>= 1;
  return c;
}

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

}  // namespace

int launch_verify_sample(const SampleLaunch& s) {
  VerifyArgs a;
  a.target = s.target;
  a.draft = s.draft;
  a.tokens = s.tokens;
  a.uniforms = s.uniforms;
  a.B = s.B;
  a.K = s.K;
  a.V = s.V;
  const double T64 = double(s.temperature);
  const double C = 1.4426950408889634073599246810018921 / T64;  // log2(e) / T
  a.C = C;
  a.c = float(C);
  a.Chi = float(C);
  a.Clo = float(C - double(a.Chi));
  const int kvec = (s.dtype == SPEC_BF16) ? 8 : 4;
  const int nvec = s.V / kvec;
  const int csize = pick_cluster(s.B, nvec);
  const int per_thread = (nvec / csize + kCons) / kCons + 1;  // vectors per thread per row slice
  a.bd.ex2 = kEx2RelErrBound;
  a.bd.gamma1 = (3.0 + per_thread + 2.0) * kUd * 1.01;
  a.bd.xbar = log2(double(s.V)) + 2.0;
  a.out_tokens = s.out_tokens;
  a.out_n = s.out_n;
  a.err = s.err;
  a.row_info = s.row_info;
  a.q_at_d = s.q_at_d;
  a.p_at_d = s.p_at_d;
  const size_t smem = smem_bytes(2 * s.K + 1);
  cudaStream_t st = static_cast<cudaStream_t>(s.stream);
  if (s.dtype == SPEC_BF16) return launch_cluster(verify_sample_kernel<EBf16>, a, s.B, csize, smem, st);
  return launch_cluster(verify_sample_kernel<EF32>, a, s.B, csize, smem, st);
}

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
  const size_t smem = smem_bytes(g.K + 1);
  cudaStream_t st = static_cast<cudaStream_t>(g.stream);
  if (g.dtype == SPEC_BF16) return launch_cluster(verify_greedy_kernel<EBf16>, a, g.B, csize, smem, st);
  return launch_cluster(verify_greedy_kernel<EF32>, a, g.B, csize, smem, st);
}

int verify_cluster_size(int B, int V, int dtype) {
  const int kvec = (dtype == SPEC_BF16) ? 8 : 4;
  return pick_cluster(B, V / kvec);
}

}  // namespace sv
