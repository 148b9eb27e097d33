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
//       finish: combine -> K accept tests -> first rejection j
//   AR  (rare) double-float sums of target and draft row i when accept test i
//       falls inside the fp32 error bound; finish: decide test i, go on
//   BS  (fallback of the bonus draw) statistics of target row K
//   SW  fp32 residual (q_j - p_j)+ over the slice of row j, re-read
//       while hot in L2, or for the bonus draw (all K accepted) the raw
//       masses 2^(z c - Kg) of target row K with an offset Kg guessed from
//       rows 0..K-1, which needs no statistics stage; per 32-vector unit
//       sums kept in the workspace; finish: locate u_K * total mass
//       slice -> unit -> entry, certify
//   FR  one pass over the draw's rows with a lighter exponential (relative
//       error < 1e-9; FD: the same pass in double-float, for the draws FR
//       cannot settle): their row sums
//       S_q, S_p and, per unit, the sums of e_q and e_p over the tokens whose
//       residual is positive. The sign of q - p = e_q/S_q - e_p/S_p is
//       decided from the fp32 normalisers with a proven margin; the few
//       tokens inside the margin are listed and decided exactly by the
//       finisher, which forms each unit's residual e_q-sum/S_q - e_p-sum/S_p
//       and runs the certified search
//   FA, FB (fallback when the list overflows) double-float row sums, then
//       the double-float residual and unit sums
// Only row j of the draft/target pair is ever re-read for the draw. The rare
// stages AR, FR, FD, FA and FB are cut finer (each slice into M pieces) so
// that a refined row's compute-heavy passes spread over more CTAs.
//
// Arithmetic. No fp64 arithmetic (GB300 runs fp64 at a small fraction of its
// fp32 rate): logits are widened to fp32, exponentials use the MUFU exp2 with
// an integer offset ceil(max * log2(e)/T), and sums a decision depends on are
// float pairs (df.cuh). A decision is taken from the fp32 path only when the
// uniform is farther from the threshold than twice a proven bound on that
// path's error; otherwise the FR stage recomputes it with a lighter
// exponential (relative error < 1e-9 per term) and, if that is not enough,
// the AR / FD / FA / FB stages with double-float exponentials (relative
// error < 4e-12 per term); the row is
// flagged in row_info. The output equals an exact-arithmetic evaluation except
// for rows flagged SPEC_ROW_UNCERTIFIED.
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

enum TaskType { kP1 = 1, kBS = 2, kSW = 3, kFA = 4, kFB = 5, kAR = 6, kFR = 7, kFD = 8 };
enum { kAccept = 0, kReject = 1, kAmbiguous = 2, kInvalid = 3 };
constexpr int kModeResidual = 0, kModeQ = 1;  // draw modes (task aux bits 8+)
constexpr int kFinWarp = kCW + 1;             // warp index of the finisher

// ------------------------------------------------------------------ arguments
struct Bounds {
  float ex2;     // relative error bound of ex2.approx.ftz.f32 on [-126, 1]
  float gamma1;  // relative error bound of the fp32 summation of row sums
  float xbar;    // bound on sum_v q_v |x_v| used by the accept tests (log2 V + 2)
};

struct SampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  int B, K, V, S, nvec;
  int M, R;        // refinement pieces per slice, per row (R = S M)
  float c;         // fl32(log2(e) / T)
  float Chi, Clo;  // log2(e) / T as a float pair
  Bounds bd;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* err;
  int32_t* row_info;
  float* q_at_d;
  float* p_at_d;
  unsigned long long* counters;  // optional acceptance statistics [2K + 2]
  const float* thr_t;            // optional [B, K + 1] target-row logit thresholds
  const float* thr_d;            // optional [B, K] draft-row logit thresholds
  int masked;                    // either is given
  // Small batches: one first-stage task per (slice, draft position), which
  // covers target and draft row i of the slice, so that the first pass
  // spreads over every CTA
  int p1sub;
  // Small batches (4 to 48 rows): a residual draw starts with FR (the
  // accurate lite pass) instead of the fp32 sweep, which leaves nearly half
  // of these draws undecided at T = 1, so that some row of the batch almost
  // surely needs the extra stage; with one to three rows the cheaper sweep
  // first is faster on average
  int direct_fr;
  Ws ws;
};

// Top-k / top-p filtering (spec_filter_thresholds): tokens whose logit is
// below their row's threshold count as logit -inf in every stage.
__device__ __forceinline__ float thr_of(const SampleArgs& a, int b, bool target, int i) {
  const float* t = target ? a.thr_t : a.thr_d;
  if (!t) return -INFINITY;
  return __ldg(t + size_t(b) * (target ? a.K + 1 : a.K) + i);
}
// Element traits plus whether the launch filters (a separate instantiation,
// so an unfiltered launch carries no compare).
template <class E0, bool M>
struct EM : E0 {
  static constexpr bool kMask = M;
};

template <int N>
__device__ __forceinline__ void mask_vals(float (&z)[N], float tau) {
#pragma unroll
  for (int k = 0; k < N; ++k) z[k] = (z[k] >= tau) ? z[k] : -INFINITY;
}

// Per-row state kept in the workspace between a row's stages. Written by the
// finisher of one stage, read (through L2) by the tasks and finisher of the
// next.
// A token whose residual sign the FR pass could not decide from the fp32
// normalisers: element index, e_q and e_p (double-float).
struct AmbEntry {
  int v, pad;
  float qh, ql, ph, pl;
};
constexpr int kAmbCap = 32;

struct RowState {
  int flags, pad0, pad1, pad2;       // SPEC_ROW_* bits so far
  float Kq, Kp, Rq, Rp;              // offsets and fp32 1/S of the draw's rows
  float Iq_hi, Iq_lo, Ip_hi, Ip_lo;  // accurate 1/S (double-float path)
  int8_t acc[32];                    // accept-test states of positions 0..K-1
  float rK[2 * kMaxK];  // offsets of rows 0..2K-1 (target i: 2i, draft i: 2i+1)
  float rR[2 * kMaxK];  // fp32 1/S of those rows
  float amb_delta;      // FR: relative margin of the fp32 sign test
  int namb;             // FR: tokens inside the margin (may exceed kAmbCap)
  int pad3, pad4;
  AmbEntry amb[kAmbCap];
};

__device__ __forceinline__ RowState* row_state(const SampleArgs& a, int b) {
  return reinterpret_cast<RowState*>(a.ws.rowstate(b));
}

// ------------------------------------------------------------------ shared memory
// Hand-off slot: the task (16 bytes), then per-warp partials.
//   P1 / BS: float wM[R][kCW], float wS[R][kCW], int wBad[R][kCW]
//   SW:      float wAcc[kCW], wAq[kCW], wAp[kCW]
//   FA / AR: df wA[kCW], wB[kCW]
//   FB:      df wR[kCW], float wQ[kCW], wP[kCW]
//   FR:      df wTq[kCW], wTp[kCW], wAq[kCW], wAp[kCW]
__host__ __device__ inline int slot_bytes(int R) {
  const int body = R * kCW * 12 > 4 * kCW * 8 ? R * kCW * 12 : 4 * kCW * 8;
  return (16 + body + 15) / 16 * 16;
}

struct Fin {  // finisher-private scratch: statistics of the 2K rows of a P1
  float rowKc[2 * kMaxK];
  df rowS[2 * kMaxK];
  df rowInv[2 * kMaxK];
  int rowOK[2 * kMaxK];
};

struct Smem {
  Ring ring;
  Handoff ho;
  Fin* fin;
  float2* tab2;  // 2^(j/256) as (hi, lo) pairs
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
  put(3, take(2 * kSlots * 8, 8));
  put(4, take(16, 16));
  put(5, take(sizeof(Fin), 16));
  put(6, take(256 * 8, 16));
  put(7, take(size_t(kSlots) * slot_bytes(R), 16));
  return al(o, 128);
}

__host__ __device__ inline size_t sample_smem_bytes(int R) { return carve(R, [](int, size_t) {}); }

__device__ inline Smem make_smem(uint8_t* base, int R) {
  Smem L;
  L.ring.buf = base;
  L.ho.slot_bytes = slot_bytes(R);
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
        L.ho.done = reinterpret_cast<uint64_t*>(p);
        L.ho.freed = L.ho.done + kSlots;
        break;
      case 4:
        L.ring.abort = reinterpret_cast<volatile int*>(p);
        break;
      case 5:
        L.fin = reinterpret_cast<Fin*>(p);
        break;
      case 6:
        L.tab2 = reinterpret_cast<float2*>(p);
        break;
      case 7:
        L.ho.data = p;
        break;
    }
  });
  return L;
}

// ------------------------------------------------------------------ statistics
// Per-thread running max M, integer offset Kc = ceil(M c) and S = sum exp2(z c - Kc).
template <class E>
struct StatOp {
  float c, M, Kc, S, tau;  // S: 1 once a term was added, else 0
  uint64_t S2;             // packed partial sums (even terms, odd terms)
  int bad;
  __device__ __forceinline__ void begin() {
    M = -INFINITY;
    Kc = -INFINITY;
    S = 0.0f;
    S2 = f2_pack(0.0f, 0.0f);
    bad = 0;
  }
  // The vectors i = tid, tid + kCons, ... < cnt of one ring stage (at most
  // kPer per thread): loaded together, one running-maximum update per stage,
  // then the exponentials, so the loads and MUFU operations overlap. The
  // exponent arguments and the sums run on packed float pairs (f32x2): the
  // running sum is a pair S2 whose halves add up the even and the odd terms
  // of each vector through a depth-2 tree, and end_row adds the halves, so
  // every term still reaches the row sum through at most 3 + run + 5 fp32
  // additions (the bound gamma1 counts).
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
      if (S != 0.0f) {
        const float sc = pow2i(__fsub_rn(Kc, Kn));
        S2 = f2_mul(S2, f2_pack(sc, sc));
        S = sc != 0.0f ? 1.0f : 0.0f;  // S only records whether any term was added
      }
      M = vm;
      Kc = Kn;
    }
    if (Kc == -INFINITY) return;  // only -inf logits so far
    const uint64_t c2 = f2_pack(c, c), nk2 = f2_pack(-Kc, -Kc);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (tid + k * kCons < cnt) {
        float z[E::kVec];
        E::unpack(v[k], z);
        if (E::kMask) mask_vals(z, tau);
        uint64_t e2[E::kVec / 2];
#pragma unroll
        for (int j = 0; j < E::kVec / 2; ++j) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(z[2 * j], z[2 * j + 1]), c2, nk2), x0, x1);
          e2[j] = f2_pack(ex2_approx(x0), ex2_approx(x1));
        }
#pragma unroll
        for (int w = 1; w < E::kVec / 2; w <<= 1)
#pragma unroll
          for (int j = 0; j < E::kVec / 2; j += 2 * w) e2[j] = f2_add(e2[j], e2[j + w]);
        S2 = f2_add(S2, e2[0]);
        S = 1.0f;
      }
    }
  }
  // Warp partial (max, sum relative to the offset of the warp's max, NaN
  // seen) of row r into the hand-off slot.
  __device__ __forceinline__ void end_row(uint8_t* slot, int R, int r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float Mw = warp_max_f(M);
    float s = 0.0f;
    if (S != 0.0f) {
      float s0, s1;
      f2_unpack(S2, s0, s1);
      s = __fmul_rn(__fadd_rn(s0, s1), pow2i(__fsub_rn(Kc, offset_of(Mw, c))));
    }
    s = warp_sum_f(s);
    const int anybad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      float* w = reinterpret_cast<float*>(slot + 16);
      w[r * kCW + warp] = Mw;
      w[(R + r) * kCW + warp] = s;
      reinterpret_cast<int*>(w + 2 * R * kCW)[r * kCW + warp] = anybad;
    }
  }
};

// ------------------------------------------------------------------ accurate path
// 2^(z C - Kc) in pair arithmetic (C = log2(e)/T as Chi + Clo, Kc an integer).
__device__ __forceinline__ df acc_elem(float z, float Chi, float Clo, float Kc,
                                       const float2* tab) {
  const df p = two_prod(z, Chi);
  const float pl = __fmaf_rn(z, Clo, p.lo);
  const df s = two_sum(p.hi, -Kc);
  return df_exp2(s.hi, __fadd_rn(s.lo, pl), tab);
}

// Relative error bound of one normalised double-float term, for a row whose
// offset is Kc: the exponential (< 4e-13 while |z C| <= 2^7; beyond, the low
// part of its argument, below 2^-23 |z C| + 2^-18, adds |t|^5/120 + 1.5 u t^2
// with |t| <= ln2 (2^-9 + 2^-23 (|Kc| + 128) + 2^-18)), its argument (< 2^-46
// (|z C| + |Kc|) with |z C| below |Kc| + 127 for every term that is not
// flushed), the normaliser sum and reciprocal (< 1e-12); kept above their
// total for every offset |Kc| < kMaxOffset = 2^18 (at 2^18 the total is 0.92
// of the bound; past about 2^18.8 the truncation would exceed it).
__device__ __forceinline__ float acc_rho(float Kc) {
  return 2e-12f + 2.2e-14f * (fabsf(Kc) + 256.0f);
}

// Relative error bound of one normalised FR term e / S: the exponential in
// the term and in each term of the normaliser (kLiteExpRelErr each), their
// pair sums (2 n^2 u^2 with n below 2^10 per thread) and the reciprocal.
constexpr float kFrRho = float(2.0 * kLiteExpRelErr + 1e-10);

// Upper bound on the sum of the computed fp32 probabilities of a row.
constexpr float kQmax = 1.001f;

// ------------------------------------------------------------------ draw entries
// fp32 path: r = max(0, q - p), q = exp2(z c - Kq) * Rq (r = q when tp is
// null). aq / ap accumulate sum q x and sum p x (x the exponent argument,
// clamped at -1e4 so that masked logits add 0), from which the error bound
// of the sweep follows.
template <class E>
struct FastEntries {
  const uint4* tq;  // rows read by entries() (the draw's search)
  const uint4* tp;
  bool pair;        // residual q - p (else q alone)
  float c, Kq, Rq, Kp, Rp;
  float tauq = -INFINITY, taup = -INFINITY;
  bool absx = false;  // aq sums q |x| (raw bonus draw) instead of q x
  // The arithmetic runs on packed float pairs (f32x2): for a residual, the
  // pair (q term, p term) of each token; for q alone, two neighbouring tokens.
  // Each half rounds exactly like the scalar operation, and the vector's sum
  // goes through a depth-3 tree as before.
  __device__ __forceinline__ float run(const uint4& vq, const uint4& vp, float (&r)[E::kVec],
                                       float& aq, float& ap) const {
    float zq[E::kVec], zp[E::kVec];
    E::unpack(vq, zq);
    if (pair) E::unpack(vp, zp);
    if (E::kMask) {
      mask_vals(zq, tauq);
      if (pair) mask_vals(zp, taup);
    }
    const uint64_t c2 = f2_pack(c, c);
    if (pair) {
      const uint64_t nk2 = f2_pack(-Kq, -Kp), r2 = f2_pack(Rq, Rp);
      uint64_t a2 = f2_pack(aq, ap);
#pragma unroll
      for (int k = 0; k < E::kVec; ++k) {
        float xa, xb;
        f2_unpack(f2_fma(f2_pack(zq[k], zp[k]), c2, nk2), xa, xb);
        float q, p;
        f2_unpack(f2_mul(f2_pack(ex2_approx(xa), ex2_approx(xb)), r2), q, p);
        a2 = f2_fma(f2_pack(q, p), f2_pack(fmaxf(xa, -1.0e4f), fmaxf(xb, -1.0e4f)), a2);
        r[k] = fmaxf(__fsub_rn(q, p), 0.0f);
      }
      f2_unpack(a2, aq, ap);
    } else {
      const uint64_t nk2 = f2_pack(-Kq, -Kq), r2 = f2_pack(Rq, Rq);
      uint64_t a2 = f2_pack(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < E::kVec; k += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(zq[k], zq[k + 1]), c2, nk2), x0, x1);
        float q0, q1;
        f2_unpack(f2_mul(f2_pack(ex2_approx(x0), ex2_approx(x1)), r2), q0, q1);
        const float w0 = fmaxf(x0, -1.0e4f), w1 = fmaxf(x1, -1.0e4f);
        a2 = f2_fma(f2_pack(q0, q1), absx ? f2_pack(fabsf(w0), fabsf(w1)) : f2_pack(w0, w1), a2);
        r[k] = q0;
        r[k + 1] = q1;
      }
      float a0, a1;
      f2_unpack(a2, a0, a1);
      aq = __fadd_rn(aq, __fadd_rn(a0, a1));
    }
    // depth-3 tree over the vector: (r0 + r1, r2 + r3) + (r4 + r5, r6 + r7), then the halves
    uint64_t t2[E::kVec / 2];
#pragma unroll
    for (int j = 0; j < E::kVec / 2; ++j) t2[j] = f2_pack(r[(j & ~1) * 2 + (j & 1)], r[(j & ~1) * 2 + (j & 1) + 2]);
    // t2[0] = (r0, r2), t2[1] = (r1, r3), t2[2] = (r4, r6), t2[3] = (r5, r7) for 8 terms
#pragma unroll
    for (int j = 0; j < E::kVec / 2; j += 2) t2[j] = f2_add(t2[j], t2[j + 1]);
#pragma unroll
    for (int w = 2; w < E::kVec / 2; w <<= 1)
#pragma unroll
      for (int j = 0; j < E::kVec / 2; j += 2 * w) t2[j] = f2_add(t2[j], t2[j + w]);
    float h0, h1;
    f2_unpack(t2[0], h0, h1);
    return __fadd_rn(h0, h1);
  }
  __device__ __forceinline__ df entries(int vi, df (&rd)[E::kVec]) const {
    float r[E::kVec];
    float a0 = 0.f, a1 = 0.f;
    const uint4 vq = ldg_nc_v4(tq + vi);
    const uint4 vp = pair ? ldg_nc_v4(tp + vi) : vq;
    const float vs = run(vq, vp, r, a0, a1);
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) rd[k] = {r[k], 0.f};
    return {vs, 0.f};
  }
};

// double-float path.
template <class E>
struct AccEntries {
  const uint4* tq;  // rows read by entries() (the draw's search)
  const uint4* tp;
  bool pair;        // residual q - p (else q alone)
  float Chi, Clo, Kq, Kp;
  df Iq, Ip;
  const float2* tab;
  float tauq = -INFINITY, taup = -INFINITY;
  __device__ __forceinline__ df run(const uint4& vq, const uint4& vp, df (&r)[E::kVec], float& qs,
                                    float& ps) const {
    float zq[E::kVec], zp[E::kVec];
    E::unpack(vq, zq);
    if (pair) E::unpack(vp, zp);
    if (E::kMask) {
      mask_vals(zq, tauq);
      if (pair) mask_vals(zp, taup);
    }
    df vs{0.f, 0.f};
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      const df q = df_mul(acc_elem(zq[k], Chi, Clo, Kq, tab), Iq);
      qs = __fadd_rn(qs, q.hi);
      df rk = q;
      if (pair) {
        const df p = df_mul(acc_elem(zp[k], Chi, Clo, Kp, tab), Ip);
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
    const uint4 vp = pair ? ldg_nc_v4(tp + vi) : vq;
    return run(vq, vp, rd, a0, a1);
  }
};

// FR's terms (lite_exp2x2, relative error < kLiteExpRelErr) normalised in
// pair arithmetic: the walk of the final unit in FR's draw, consistent with
// the unit sums of the FR pass.
template <class E>
struct LiteEntries {
  const uint4* tq;
  const uint4* tp;
  bool pair;
  LiteConsts LC;
  LiteRow Lq, Lp;
  df Iq, Ip;
  const float2* tab;
  float tauq = -INFINITY, taup = -INFINITY;
  __device__ __forceinline__ df entries(int vi, df (&rd)[E::kVec]) const {
    const uint4 vq = ldg_nc_v4(tq + vi);
    const uint4 vp = pair ? ldg_nc_v4(tp + vi) : vq;
    float zq[E::kVec], zp[E::kVec];
    E::unpack(vq, zq);
    if (pair) E::unpack(vp, zp);
    if (E::kMask) {
      mask_vals(zq, tauq);
      if (pair) mask_vals(zp, taup);
    }
    df vs{0.f, 0.f};
    if (pair) {
#pragma unroll
      for (int k = 0; k < E::kVec; ++k) {
        df eq, ep;
        lite_exp2x2(zq[k], zp[k], Lq, Lp, LC, tab, eq, ep);
        df rk = df_sub(df_mul(eq, Iq), df_mul(ep, Ip));
        if (!(rk.hi > 0.0f)) rk = {0.f, 0.f};
        rd[k] = rk;
        vs = df_add(vs, rk);
      }
    } else {
#pragma unroll
      for (int k = 0; k < E::kVec; k += 2) {
        df e0, e1;
        lite_exp2x2(zq[k], zq[k + 1], Lq, Lq, LC, tab, e0, e1);
        rd[k] = df_mul(e0, Iq);
        rd[k + 1] = df_mul(e1, Iq);
        vs = df_add(df_add(vs, rd[k]), rd[k + 1]);
      }
    }
    return vs;
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

// Rows of a draw stage (SW, FA, FB) from the task's aux: target row j and,
// for a residual draw before the bonus position, draft row j.
struct DrawRows {
  int j;
  bool pair;
};
__device__ __forceinline__ DrawRows draw_rows(int K, int aux) {
  const int j = aux & 0xff, mode = (aux >> 8) & 1;
  return {j, mode == kModeResidual && j < K};
}

// The rare stages AR, FA and FB may run on pieces instead of slices (task aux
// bit kPieceBit): the finisher that enqueues them chooses pieces once every
// first-stage task is claimed, when the launch's tail has idle CTAs and few
// runnable tasks; before that whole slices keep the task count low.
constexpr int kPieceBit = 1 << 9;
// The bonus draw from q_K without a statistics stage (task aux bit kRawBit):
// the sweep sums e = 2^(z c - Kg) with a guessed offset Kg (the largest of
// target rows 0..K-1's) and the draw compares u_K times their total with
// their prefix sums, so no normaliser enters; a total that is not finite or
// below 2^-60 (the guess far off) sends the row to the statistics stage BS.
constexpr int kRawBit = 1 << 10;

__device__ __forceinline__ bool is_piece(const QTask& t) {
  return (t.type == kAR || t.type == kFA || t.type == kFB || t.type == kFR || t.type == kFD) &&
         (t.aux & kPieceBit);
}

// kPieceBit if the next rare stage of a row should run on pieces.
__device__ __forceinline__ int piece_choice(const SampleArgs& a) {
  if (a.M == 1) return 0;
  return ld_volatile_u32(&a.ws.hdr()->p1_next) >=
                 uint32_t(a.B) * uint32_t(a.S) * uint32_t(a.p1sub ? a.K : 1)
             ? kPieceBit
             : 0;
}

__device__ __forceinline__ int stage_tasks(const SampleArgs& a, int piece_bit) {
  return piece_bit ? a.R : a.S;
}

// Queues a rare stage of row b (all lanes; lane 0's arguments), on slices or
// pieces as piece_choice decides.
__device__ __forceinline__ void enqueue_rare(const SampleArgs& a, int type, int b, int aux) {
  const int pb = __shfl_sync(0xffffffffu, (threadIdx.x & 31) == 0 ? piece_choice(a) : 0, 0);
  enqueue_row_stage(a.ws, type, b, stage_tasks(a, pb), aux | pb);
}

// Vector range [v0, v1) of the task's part of the row: slice s, or for the
// piece stages piece s (slice s / M cut into M runs of whole 32-vector units,
// none empty since a slice has at least M units). pv0 is the start of the
// enclosing slice, whose unit-sum array the piece writes into.
__device__ __forceinline__ void task_range(const SampleArgs& a, bool pieces, int s, int& v0,
                                           int& v1, int& ps, int& pv0) {
  if (!pieces) {
    slice_range(a.nvec, a.S, s, v0, v1);
    ps = s;
    pv0 = v0;
    return;
  }
  ps = s / a.M;
  const int i = s % a.M;
  int s0, s1;
  slice_range(a.nvec, a.S, ps, s0, s1);
  const int units = (s1 - s0 + 31) / 32;
  v0 = s0 + (units * i / a.M) * 32;
  v1 = (i == a.M - 1) ? s1 : s0 + (units * (i + 1) / a.M) * 32;
  pv0 = s0;
}

// Partials of piece p of row b (8 floats) inside the row's partial block.
__device__ __forceinline__ float* piece_part(const SampleArgs& a, int b, int p) {
  return a.ws.part(b, 0) + 8 * p;
}

// Partials of a task's slice or piece.
__device__ __forceinline__ float* task_part(const SampleArgs& a, bool pieces, int b, int s) {
  return pieces ? piece_part(a, b, s) : a.ws.part(b, s);
}

// ------------------------------------------------------------------ finisher
// Everything below runs in the finisher warp (32 lanes). Data written by
// other CTAs (partials, unit sums, row state) is read through L2 (ld.cg).

// Row statistics of rows [0, nrows) (float offset 4r of each slice's
// partials: max, sum hi, sum lo, NaN seen) into the finisher scratch. Rows
// are taken up to 32 at a time; each row gets g lanes (g = 32 / rows, a
// power of two), lane k of a row combines slices k, k + g, ... in batches of
// kStatBatch loads issued together (one memory round trip per batch), keeping
// a running offset: a larger maximum rescales the running sum by the power of
// two between the offsets, which is exact, so the sum equals the one taken
// at the final offset term by term (up to terms below 2^-126 of the
// largest). The row's lanes then merge with g / 2 .. 1 butterfly shuffles.
constexpr int kStatBatch = 8;
__device__ void stats_rows(const SampleArgs& a, Fin& F, int b, int nrows) {
  const int lane = threadIdx.x & 31, S = a.S;
  for (int r0 = 0; r0 < nrows; r0 += 32) {
    const int rg = min(32, nrows - r0);
    int g = 1;
    while (g * 2 * rg <= 32) g *= 2;
    const int rr = lane / g, k = lane % g, r = r0 + rr;
    const bool live = rr < rg;
    float M = -INFINITY, Kr = -INFINITY;  // running maximum and its offset
    df Ssum{0.f, 0.f};                    // at offset Kr
    int bad = 0;
    for (int s0 = k; s0 < S; s0 += kStatBatch * g) {
      float4 it[kStatBatch];
#pragma unroll
      for (int q = 0; q < kStatBatch; ++q) {
        const int sl = s0 + q * g;
        it[q] = (live && sl < S) ? __ldcg(reinterpret_cast<const float4*>(a.ws.part(b, sl) + 4 * r))
                                 : make_float4(-INFINITY, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < kStatBatch; ++q) {
        M = fmaxf(M, it[q].x);
        bad |= __float_as_int(it[q].w);
      }
      const float Kn = offset_of(M, a.c);
      if (Kn > Kr) {
        if (Ssum.hi != 0.0f) {
          const float sc = pow2i(__fsub_rn(Kr, Kn));
          Ssum = df{__fmul_rn(Ssum.hi, sc), __fmul_rn(Ssum.lo, sc)};
        }
        Kr = Kn;
      }
#pragma unroll
      for (int q = 0; q < kStatBatch; ++q) {
        if (it[q].y != 0.0f) {
          const float sc = pow2i(__fsub_rn(offset_of(it[q].x, a.c), Kr));
          Ssum = df_add(Ssum, df{__fmul_rn(it[q].y, sc), __fmul_rn(it[q].z, sc)});
        }
      }
    }
    for (int o = g / 2; o > 0; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    const float Kc = offset_of(M, a.c);
    if (Ssum.hi != 0.0f) {  // to the row's offset (Kr <= Kc, both finite here)
      const float sc = pow2i(__fsub_rn(Kr, Kc));
      Ssum = df{__fmul_rn(Ssum.hi, sc), __fmul_rn(Ssum.lo, sc)};
    }
    for (int o = g / 2; o > 0; o >>= 1) Ssum = df_add(Ssum, df_shfl_xor(Ssum, o));
    if (live && k == 0) {
      const bool ok = !bad && isfinite(M) && fabsf(Kc) < kMaxOffset && Ssum.hi > 0.0f &&
                      isfinite(Ssum.hi);
      F.rowKc[r] = Kc;
      F.rowS[r] = Ssum;
      F.rowInv[r] = ok ? df_recip(Ssum) : df{0.f, 0.f};
      F.rowOK[r] = ok ? 1 : 0;
    }
    __syncwarp();
  }
}

// Sums over the slices (or pieces) of the four floats of their partials, lanes
// in parallel: x0 + x1 as a pair, x2 and x3 as floats (or x2 + x3 as a
// second pair when `pairs`). Every lane gets the totals.
struct SliceSums {
  df p0, p1;
  float f2, f3;
};
__device__ SliceSums slice_sums(const SampleArgs& a, int b, bool pairs, bool pieces) {
  const int lane = threadIdx.x & 31;
  df p0{0.f, 0.f}, p1{0.f, 0.f};
  float f2 = 0.f, f3 = 0.f;
  for (int sl = lane; sl < (pieces ? a.R : a.S); sl += 32) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(task_part(a, pieces, b, sl)));
    p0 = df_add(p0, df{v.x, v.y});
    if (pairs) {
      p1 = df_add(p1, df{v.z, v.w});
    } else {
      f2 += v.z;
      f3 += v.w;
    }
  }
  SliceSums r;
  r.p0 = df_warp_sum(p0);
  r.p1 = pairs ? df_warp_sum(p1) : df{0.f, 0.f};
  r.f2 = warp_sum_f(f2);
  r.f3 = warp_sum_f(f3);
  return r;
}

// Writes row b's outputs: accepted tokens 0..n-1 (lane i holds draft token i
// in `tok`), `token` at n, -1 after (all -1 on error), num_accepted and
// row_info; counts the row done. The count only lets the producers stop, so
// no fence orders the outputs before it (the launch's end publishes them).
__device__ void write_outputs(const SampleArgs& a, int b, int n, int token, int flags, bool error,
                              int tok) {
  const int lane = threadIdx.x & 31, K = a.K;
  if (lane <= K) {
    int32_t v;
    if (error) v = -1;
    else if (lane < n) v = tok;
    else if (lane == n) v = token;
    else v = -1;
    a.out_tokens[size_t(b) * (K + 1) + lane] = v;
  }
  if (lane == 0) {
    a.out_n[b] = error ? -1 : n;
    if (a.row_info) a.row_info[b] = flags;
    atomicAdd(&a.ws.hdr()->rows_done, 1u);
  }
  if (a.counters && !error) count_acceptance(a.counters, K, n);
  __syncwarp();
}

// Draft tokens of row b, lane i holding position i (0 past K).
__device__ __forceinline__ int load_tokens(const SampleArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  return lane < a.K ? a.tokens[size_t(b) * a.K + lane] : 0;
}

// Starts the draw at position j: the residual of target / draft row j with
// the fp32 statistics given (lane 0's values), or (j == K) the bonus
// distribution q_K, drawn without its statistics (kRawBit) with the offset
// guessed from target rows 0..K-1.
__device__ void start_draw(const SampleArgs& a, int b, int j, int flags, float Kq, float Rq,
                           float Kp, float Rp) {
  const int lane = threadIdx.x & 31;
  RowState* st = row_state(a, b);
  float Kg = 0.f;
  if (j == a.K) {
    __syncwarp();  // orders finish_p1's stores of the row offsets
    Kg = warp_max_f(lane < a.K ? __ldcg(&st->rK[2 * lane]) : -INFINITY);
  }
  const bool fr = j < a.K && a.direct_fr && fabsf(Kq) <= kLiteMaxOffset &&
                  fabsf(Kp) <= kLiteMaxOffset;
  if (lane == 0) {
    st->flags = flags;
    if (j < a.K) {
      st->Kq = Kq;
      st->Rq = Rq;
      st->Kp = Kp;
      st->Rp = Rp;
    } else {
      st->Kq = Kg;
      st->Rq = 1.0f;  // the raw sweep sums e, not q
    }
    if (fr) {
      // FR's sign-test margin as after the sweep (finish_sw), with the sums
      // q|x| and p|x| bounded by xbar instead of measured
      const float eps = a.bd.ex2 + a.bd.gamma1 +
                        2.0f * kLn2f * kU * (1.01f * a.bd.xbar + 0.5f * kQmax) + 4.0f * kU +
                        float(kLiteExpRelErr);
      st->amb_delta = 1.05f * 2.0f * eps + 4.0f * kU;
      st->namb = 0;
    }
  }
  if (fr) {
    enqueue_rare(a, kFR, b, j | (kModeResidual << 8));
    return;
  }
  enqueue_row_stage(a.ws, kSW, b, a.S,
                    j < a.K ? (j | (kModeResidual << 8)) : (a.K | (kModeQ << 8) | kRawBit));
}

// Continues the accept tests from position i0 given the test states (lane i
// holds test i's state in `state`, its offsets / fp32 1/S of target and
// draft row i in rk_t, rr_t, rk_d, rr_d): skips accepted positions and stops
// at a rejection (draw), an invalid row (error), an ambiguous test (AR
// stage) or the end (bonus draw).
__device__ void continue_tests(const SampleArgs& a, int b, int i0, int flags, int state, int tok,
                               float rk_t, float rr_t, float rk_d, float rr_d) {
  const int lane = threadIdx.x & 31, K = a.K;
  const unsigned pend = __ballot_sync(0xffffffffu, lane >= i0 && lane < K && state != kAccept);
  if (!pend) {
    start_draw(a, b, K, flags, 0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int i = __ffs(int(pend)) - 1;
  const int s = __shfl_sync(0xffffffffu, state, i);
  if (s == kReject) {
    start_draw(a, b, i, flags, __shfl_sync(0xffffffffu, rk_t, i), __shfl_sync(0xffffffffu, rr_t, i),
               __shfl_sync(0xffffffffu, rk_d, i), __shfl_sync(0xffffffffu, rr_d, i));
    return;
  }
  if (s == kInvalid) {
    if (lane == 0 && a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
    write_outputs(a, b, i, -1, flags, true, tok);
    return;
  }
  // ambiguous: double-float sums of target and draft row i (AR stage)
  if (lane == 0) row_state(a, b)->flags = flags | SPEC_ROW_ACCEPT_REFINED;
  enqueue_rare(a, kAR, b, i);
}

// P1 complete: statistics of the 2K rows, accept tests, first rejection.
// Memory round trips: the draft tokens and uniforms; then the logits at the
// draft tokens together with the first batch of slice partials; then any
// further batches of partials.
template <class E>
__device__ void finish_p1(const SampleArgs& a, const Smem& L, int b) {
  const int lane = threadIdx.x & 31, K = a.K, V = a.V;
  Fin& F = *L.fin;
  RowState* st = row_state(a, b);
  const RowPtrs<E> rp = row_ptrs<E>(a, b);
  const int d = load_tokens(a, b);
  const float u = lane < K ? a.uniforms[size_t(b) * (K + 1) + lane] : 1.0f;
  const bool badtok_lane = lane < K && (d < 0 || d >= V);
  // raw elements: converted only after the statistics, so that nothing
  // waits for these loads before the partials' loads are issued
  typename E::T rt{}, rd{};
  if (lane < K && !badtok_lane) {
    rt = rp.tgt[size_t(lane) * V + d];
    rd = rp.drf[size_t(lane) * V + d];
  }
  stats_rows(a, F, b, 2 * K);
  float zt = E::cvt(rt), zd = E::cvt(rd);
  if (E::kMask && lane < K && !badtok_lane) {
    if (!(zt >= thr_of(a, b, true, lane))) zt = -INFINITY;
    if (!(zd >= thr_of(a, b, false, lane))) zd = -INFINITY;
  }
  for (int r = lane; r < 2 * K; r += 32) {
    st->rK[r] = F.rowKc[r];
    st->rR[r] = F.rowInv[r].hi;
  }
  const float c = a.c;
  int s = kAccept;
  float rk_t = 0.f, rr_t = 0.f, rk_d = 0.f, rr_d = 0.f;
  if (lane < K) {
    const int rt = 2 * lane, rd = 2 * lane + 1;
    rk_t = F.rowKc[rt];
    rr_t = F.rowInv[rt].hi;
    rk_d = F.rowKc[rd];
    rr_d = F.rowInv[rd].hi;
    float qd = -1.f, pd = -1.f;
    if (badtok_lane || !F.rowOK[rt] || !F.rowOK[rd]) {
      s = kInvalid;
    } else {
      const float xt = __fmaf_rn(zt, c, -rk_t);
      const float xd = __fmaf_rn(zd, c, -rk_d);
      qd = __fmul_rn(ex2_approx(xt), rr_t);
      pd = __fmul_rn(ex2_approx(xd), rr_d);
      if (zd == -INFINITY) {
        s = kAccept;  // p(d) = 0 accepts
      } else if (zt == -INFINITY) {
        s = kReject;  // q(d) = 0: u < 0 never holds
      } else if (u == 0.0f) {
        s = kAccept;  // 0 < q(d)/p(d) whenever q(d) > 0
      } else {
        // ratio = 2^(xt - xd) * S_d / S_t; relative error bound: exp2, the
        // arguments (with the fp32 temperature constant), both row sums and
        // five roundings
        const float ar = __fsub_rn(xt, xd);
        const float ratio = __fmul_rn(__fmul_rn(ex2_approx(ar), F.rowS[rd].hi), rr_t);
        const float dS = a.bd.ex2 + kLn2f * kU * a.bd.xbar + a.bd.gamma1;
        const float beta =
            1.1f * (a.bd.ex2 + 6.0f * kU + 2.0f * dS +
                    kLn2f * kU * (2.0f * fabsf(xt) + 2.0f * fabsf(xd) + fabsf(ar) +
                                  2.0f * a.bd.xbar + 4.0f));
        if (!(ar < 126.0f) || ratio >= 1.0f / (1.0f - beta)) {
          s = kAccept;  // ratio >= 1 for certain
        } else {
          const float rlo = fminf(1.0f, __fmul_rn(ratio, 1.0f - beta));
          const float rhi = fminf(1.0f, __fmul_rn(ratio, 1.0f + beta));
          s = (u < rlo) ? kAccept : (u >= rhi && ar > -120.0f ? kReject : kAmbiguous);
        }
      }
    }
    st->acc[lane] = int8_t(s);
    if (a.q_at_d) {
      a.q_at_d[size_t(b) * K + lane] = qd;
      a.p_at_d[size_t(b) * K + lane] = pd;
    }
  }
  if (__any_sync(0xffffffffu, badtok_lane)) {
    if (lane == 0 && a.err) atomicOr(a.err, SPEC_DERR_TOKEN);
    write_outputs(a, b, 0, -1, 0, true, d);
    return;
  }
  continue_tests(a, b, 0, 0, s, d, rk_t, rr_t, rk_d, rr_d);
}

// AR complete: decide accept test i from double-float row sums.
template <class E>
__device__ void finish_ar(const SampleArgs& a, const Smem& L, int b, int aux) {
  const int lane = threadIdx.x & 31, K = a.K, i = aux & 0xff;
  RowState* st = row_state(a, b);
  const int d = load_tokens(a, b);
  int state = kAccept;
  float rk_t = 0.f, rr_t = 0.f, rk_d = 0.f, rr_d = 0.f;
  if (lane < K) {
    state = __ldcg(&st->acc[lane]);
    rk_t = __ldcg(&st->rK[2 * lane]);
    rr_t = __ldcg(&st->rR[2 * lane]);
    rk_d = __ldcg(&st->rK[2 * lane + 1]);
    rr_d = __ldcg(&st->rR[2 * lane + 1]);
  }
  int flags = __ldcg(&st->flags);
  const float u = a.uniforms[size_t(b) * (K + 1) + i];
  const SliceSums ss = slice_sums(a, b, true, aux & kPieceBit);
  const df S0 = ss.p0, S1 = ss.p1;
  const RowPtrs<E> rp = row_ptrs<E>(a, b);
  const int di = __shfl_sync(0xffffffffu, d, i);
  float zt = E::load(rp.tgt + size_t(i) * a.V, di);
  float zd = E::load(rp.drf + size_t(i) * a.V, di);
  if (E::kMask) {
    if (!(zt >= thr_of(a, b, true, i))) zt = -INFINITY;
    if (!(zd >= thr_of(a, b, false, i))) zd = -INFINITY;
  }
  // ratio = 2^((zt C - Kt) - (zd C - Kd)) * S_d / S_t in pair arithmetic
  const df xt = df_add_f(df_add(two_prod(zt, a.Chi), df{__fmul_rn(zt, a.Clo), 0.f}),
                         -__shfl_sync(0xffffffffu, rk_t, i));
  const df xd = df_add_f(df_add(two_prod(zd, a.Chi), df{__fmul_rn(zd, a.Clo), 0.f}),
                         -__shfl_sync(0xffffffffu, rk_d, i));
  const df ar = df_sub(xt, xd);
  bool acc;
  if (ar.hi >= 127.0f) {
    acc = true;
  } else if (ar.hi < -126.0f) {
    acc = false;  // ratio < 2^-100 < u (u > 0 here)
  } else {
    const df ratio = df_mul(df_mul(df_exp2(ar.hi, ar.lo, L.tab2), S1), df_recip(S0));
    acc = (ratio.hi >= 1.0f) || df_gt(ratio, df{u, 0.f});
    if (fabsf(__fsub_rn(u, fminf(1.0f, ratio.hi))) <= 1e-10f * ratio.hi)
      flags |= SPEC_ROW_UNCERTIFIED;
  }
  if (acc) {
    if (lane == i) {
      state = kAccept;
      st->acc[i] = kAccept;
    }
    continue_tests(a, b, i + 1, flags, state, d, rk_t, rr_t, rk_d, rr_d);
  } else {
    start_draw(a, b, i, flags, __shfl_sync(0xffffffffu, rk_t, i), __shfl_sync(0xffffffffu, rr_t, i),
               __shfl_sync(0xffffffffu, rk_d, i), __shfl_sync(0xffffffffu, rr_d, i));
  }
}

// BS complete: statistics of target row K, then the bonus draw.
__device__ void finish_bs(const SampleArgs& a, const Smem& L, int b) {
  const int lane = threadIdx.x & 31;
  Fin& F = *L.fin;
  RowState* st = row_state(a, b);
  const int flags = __ldcg(&st->flags);
  stats_rows(a, F, b, 1);
  if (!F.rowOK[0]) {
    const int d = load_tokens(a, b);
    if (lane == 0 && a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
    write_outputs(a, b, a.K, -1, flags, true, d);
    return;
  }
  if (lane == 0) {
    st->Kq = F.rowKc[0];
    st->Rq = F.rowInv[0].hi;
  }
  enqueue_row_stage(a.ws, kSW, b, a.S, a.K | (kModeQ << 8));
}

// The segment sums of a draw stage (slices after SW, pieces after FB), lanes
// in parallel: lane l holds segments l and l + 32 (x0 + x1 as a pair in xa /
// xb, the other two floats in f2 / f3), and the row totals (every lane).
struct DrawSlices {
  df xa, xb;  // this lane's segments
  df total;
  float f2, f3;
  bool pieces;
  int n;  // segments
};
__device__ DrawSlices draw_slices(const SampleArgs& a, int b, bool pieces) {
  const int lane = threadIdx.x & 31;
  DrawSlices r;
  r.pieces = pieces;
  r.n = pieces ? a.R : a.S;
  r.xa = r.xb = df{0.f, 0.f};
  float f2 = 0.f, f3 = 0.f;
  auto seg = [&](int i) { return pieces ? piece_part(a, b, i) : a.ws.part(b, i); };
  if (lane < r.n) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(seg(lane)));
    r.xa = df{v.x, v.y};
    f2 = v.z;
    f3 = v.w;
  }
  if (lane + 32 < r.n) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(seg(lane + 32)));
    r.xb = df{v.x, v.y};
    f2 += v.z;
    f3 += v.w;
  }
  r.total = df_warp_sum(df_add(r.xa, r.xb));
  r.f2 = warp_sum_f(f2);
  r.f3 = warp_sum_f(f3);
  return r;
}

// Unit sums as stored by SW and FB: one pair per unit.
struct PlainUnits {
  const SampleArgs* a;
  int b;
  // unit `u` of slice `ps` (index from the slice start); all lanes call it
  __device__ __forceinline__ df get(int ps, int u, bool valid) const {
    if (!valid) return df{0.f, 0.f};
    const float2 w = __ldcg(a->ws.units(b, ps) + u);
    return df{w.x, w.y};
  }
};

// Locates t in the row's draw entries: the slice (from the lanes' slice
// sums), then the 32-vector unit, then the entry (the warp walks the unit).
// Returns the token (-1 if none) and whether it is certified: both
// boundaries of the drawn entry farther than 2.02 E from t.
template <class E, class Entries, class Units>
__device__ int search_draw(const SampleArgs& a, int b, const Entries& ent, const DrawSlices& sl,
                           df t, float Eb, bool& cert, const Units& units_src) {
  const int lane = threadIdx.x & 31;
  // slice: lanes scan 32 slices at a time; the first slice with mass whose
  // end passes t, else the last slice with mass (rounding fallback)
  int ss = -1;
  df pre_s{0.f, 0.f};
  {
    df sbase{0.f, 0.f};
    for (int s0 = 0; s0 < sl.n; s0 += 32) {
      const df x = (s0 == 0) ? sl.xa : sl.xb;
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
    int v0, v1, ps, pv0;
    task_range(a, sl.pieces, ss, v0, v1, ps, pv0);
    const int nu = (v1 - v0 + 31) / 32;
    // unit: lanes scan 32 units at a time
    const int ub = (v0 - pv0) / 32;
    int us = -1;
    df ubase = pre_s, ubase_s = pre_s;
    // the unit sums of up to kPre passes are loaded together (one memory
    // round trip), then scanned pass by pass
    constexpr int kPre = 2;
    for (int g0 = 0; g0 < nu && us < 0; g0 += 32 * kPre) {
     df xs[kPre];
#pragma unroll
     for (int p = 0; p < kPre; ++p) {
       const int u = g0 + 32 * p + lane;
       xs[p] = units_src.get(ps, ub + u, u < nu);
     }
#pragma unroll
     for (int p = 0; p < kPre; ++p) {
      const int u0 = g0 + 32 * p;
      if (u0 >= nu || us >= 0) break;
      const int u = u0 + lane;
      const df x = xs[p];
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
  const float m1 = df_sub(t, tlo).hi, m2 = df_sub(thi, t).hi;
  cert = token >= 0 && fminf(m1, m2) > 2.02f * Eb;
  return token;
}

// SW complete: fp32 draw with its error bound; certified, or on to FA.
template <class E>
__device__ void finish_sw(const SampleArgs& a, int b, int aux) {
  const int lane = threadIdx.x & 31;
  RowState* st = row_state(a, b);
  const DrawRows dr = draw_rows(a.K, aux);
  const int d = load_tokens(a, b);
  const int flags = __ldcg(&st->flags);
  const float Kq = __ldcg(&st->Kq), Rq = __ldcg(&st->Rq);
  const float Kp = dr.pair ? __ldcg(&st->Kp) : 0.f, Rp = dr.pair ? __ldcg(&st->Rp) : 0.f;
  const float uK = a.uniforms[size_t(b) * (a.K + 1) + a.K];
  const DrawSlices sl = draw_slices(a, b, false);
  const df Sr = sl.total;
  const bool raw = (aux & kRawBit) != 0;
  if (raw && !(Sr.hi > 8.6736174e-19f && Sr.hi < 1.2676506e30f)) {
    // the guessed offset is far off (total below 2^-60 or above 2^100, or not
    // finite): the statistics stage, then the normalised draw. Below 2^100
    // every exponent argument is below 100, inside the range over which the
    // ex2 bound is measured, and the sweep's sum of q|x| stays finite.
    enqueue_row_stage(a.ws, kBS, b, a.S, a.K | (kModeQ << 8));
    return;
  }
  // Error bound (probability units) of the fp32 sweep. Per term, relative:
  // exp2 (ex2), argument rounding and the fp32 temperature constant (ln2 u |x|
  // each), 1/S and the product (3u), and the row sum behind 1/S (ex2 + ln2 u
  // sum q|x| + gamma1); summed with weights q (resp. p), whose sum is at most
  // kQmax. sum q|x| <= kQmax/2 - sum q x, since x <= 1/4 (the offset is the
  // ceiling of the rounded max * c, below 2^18 in magnitude). Summation: each
  // term reaches a unit sum through the 8-term vector tree and the 32-lane
  // warp tree (gamma_8), and every unit, slice and row sum above that is pair
  // arithmetic, so t and each computed boundary are within about 8.1 u Sr of
  // their exact sums over the computed terms; 16 u Sr covers that.
  auto side = [&](float A) {
    const float absx = 1.01f * fmaxf(0.0f, -A) + 0.5f * kQmax;
    return 1.05f * (kQmax * (2.0f * a.bd.ex2 + 3.0f * kU + a.bd.gamma1 + 4.0f * kLn2f * kU) +
                    4.0f * kLn2f * kU * absx);
  };
  // Raw bonus draw (units of e, total Sr): t = u_K Sr and every boundary are
  // sums of the same computed terms, so a factor common to all terms cancels
  // and no normaliser enters. Per term, relative: exp2 (ex2) and the argument
  // and temperature-constant roundings (ln2 u |x| each; the constant's part
  // common to all terms cancels); weights q = e / Sr, sum q|x| from the sweep
  // (x may be positive here: the offset is a guess).
  auto side_raw = [&](float A) {
    const float absx = 1.01f * A / Sr.hi + 1e-6f;
    return Sr.hi * 1.05f * (kQmax * (a.bd.ex2 + 3.0f * kU + 4.0f * kLn2f * kU) +
                            2.0f * kLn2f * kU * absx);
  };
  const float Eb = (raw ? side_raw(sl.f2) : side(sl.f2) + (dr.pair ? side(sl.f3) : 0.f)) +
                   16.0f * kU * Sr.hi + 1e-30f;
  const df t = df_mul_f(Sr, uK);
  int token = -1;
  bool cert = false;
  if (Sr.hi > 2.0f * Eb) {
    const RowPtrs<E> rp = row_ptrs<E>(a, b);
    FastEntries<E> fe;
    fe.tq = reinterpret_cast<const uint4*>(rp.tgt + size_t(dr.j) * a.V);
    fe.tp = dr.pair ? reinterpret_cast<const uint4*>(rp.drf + size_t(dr.j) * a.V) : nullptr;
    fe.pair = dr.pair;
    fe.c = a.c;
    fe.tauq = thr_of(a, b, true, dr.j);
    fe.taup = dr.pair ? thr_of(a, b, false, dr.j) : -INFINITY;
    fe.Kq = Kq;
    fe.Rq = Rq;
    fe.Kp = Kp;
    fe.Rp = Rp;
    token = search_draw<E>(a, b, fe, sl, t, Eb, cert, PlainUnits{&a, b});
  }
  if (token >= 0 && cert) {
    write_outputs(a, b, dr.j, token, flags, false, d);
    return;
  }
  if (lane == 0) {
    // FR's sign test compares fp32 approximations x = e_q.hi * Rq and
    // y = e_p.hi * Rp of q and p. Relative error of each: the fp32 row sum
    // behind R (ex2 + gamma1 + 2 ln2 u sum q|x|), the reciprocal, the hi
    // part and the product (about 3u), and FR's exponential (kLiteExpRelErr).
    auto eps = [&](float A) {
      const float absx = 1.01f * fmaxf(0.0f, -A) + 0.5f * kQmax;
      return a.bd.ex2 + a.bd.gamma1 + 2.0f * kLn2f * kU * absx + 4.0f * kU +
             float(kLiteExpRelErr);
    };
    st->amb_delta = 1.05f * (eps(sl.f2) + eps(sl.f3)) + 4.0f * kU;
    st->namb = 0;
    st->flags = flags | SPEC_ROW_SAMPLE_REFINED;
  }
  // FR's exponential needs offsets within kLiteMaxOffset; beyond, the
  // double-float pass FD refines the draw
  const bool lite = fabsf(Kq) <= kLiteMaxOffset && (!dr.pair || fabsf(Kp) <= kLiteMaxOffset);
  enqueue_rare(a, lite ? kFR : kFD, b, aux & ~kPieceBit);
}

// Element index (token) of an ambiguous FR entry -> its slice or piece.
__device__ __forceinline__ int part_of_token(const SampleArgs& a, bool pieces, int v) {
  const int vv = v / (a.V / a.nvec);
  int s = int(int64_t(vv) * a.S / a.nvec);
  int s0, s1;
  slice_range(a.nvec, a.S, s, s0, s1);
  while (s > 0 && vv < s0) slice_range(a.nvec, a.S, --s, s0, s1);
  while (s < a.S - 1 && vv >= s1) slice_range(a.nvec, a.S, ++s, s0, s1);
  if (!pieces) return s;
  const int units = (s1 - s0 + 31) / 32, uu = (vv - s0) / 32;
  int i = 0;
  while (i < a.M - 1 && uu >= units * (i + 1) / a.M) ++i;
  return s * a.M + i;
}

// FR unit values: residual of unit u = Aq_u / S_q - Ap_u / S_p plus the
// positive ambiguous tokens inside it (held one per lane: token av, value ad).
struct FrUnits {
  const SampleArgs* a;
  int b, namb, av;
  bool pair;
  df Iq, Ip, ad;
  __device__ __forceinline__ df get(int ps, int u, bool valid) const {
    df x{0.f, 0.f};
    if (valid) {
      const float4 w = __ldcg(reinterpret_cast<const float4*>(a->ws.units(b, ps)) + u);
      x = df_mul(df{w.x, w.y}, Iq);
      if (pair) x = df_sub(x, df_mul(df{w.z, w.w}, Ip));
    }
    if (namb > 0) {
      int s0, s1;
      slice_range(a->nvec, a->S, ps, s0, s1);
      const int kv = a->V / a->nvec;
      const int e0 = (s0 + 32 * u) * kv, e1 = e0 + 32 * kv;
      for (int e = 0; e < namb; ++e) {
        const int ve = __shfl_sync(0xffffffffu, av, e);
        const df de = df_shfl(ad, e);
        if (valid && ve >= e0 && ve < e1) x = df_add(x, de);
      }
    }
    return x;
  }
};

// FA complete: accurate normalisers of the draw's rows, then FB.
__device__ void finish_fa(const SampleArgs& a, int b, int aux) {
  const int lane = threadIdx.x & 31;
  const DrawRows dr = draw_rows(a.K, aux);
  const SliceSums ss = slice_sums(a, b, true, aux & kPieceBit);
  if (lane == 0) {
    RowState* st = row_state(a, b);
    const df I0 = df_recip(ss.p0);
    st->Iq_hi = I0.hi;
    st->Iq_lo = I0.lo;
    if (dr.pair) {
      const df I1 = df_recip(ss.p1);
      st->Ip_hi = I1.hi;
      st->Ip_lo = I1.lo;
    }
  }
  enqueue_rare(a, kFB, b, aux & ~kPieceBit);
}

// FB complete: certified double-float draw (or the zero-residual rerun on q_j).
template <class E>
__device__ void finish_fb(const SampleArgs& a, const Smem& L, int b, int aux) {
  const int lane = threadIdx.x & 31;
  RowState* st = row_state(a, b);
  const DrawRows dr = draw_rows(a.K, aux);
  const int d = load_tokens(a, b);
  const int flags = __ldcg(&st->flags);
  const float Kq = __ldcg(&st->Kq), Kp = dr.pair ? __ldcg(&st->Kp) : 0.f;
  const df Iq{__ldcg(&st->Iq_hi), __ldcg(&st->Iq_lo)};
  const df Ip = dr.pair ? df{__ldcg(&st->Ip_hi), __ldcg(&st->Ip_lo)} : df{0.f, 0.f};
  const float uK = a.uniforms[size_t(b) * (a.K + 1) + a.K];
  const DrawSlices sl = draw_slices(a, b, aux & kPieceBit);
  const df Sr = sl.total;
  const float Eb = fmaxf(acc_rho(Kq), acc_rho(Kp)) * (sl.f2 + sl.f3) + 1e-14f * Sr.hi + 1e-36f;
  if (!(Sr.hi > 0.0f) && dr.pair) {
    // zero residual mass: the draw uses q_j itself
    if (lane == 0) st->flags = flags | SPEC_ROW_ZERO_RESIDUAL;
    enqueue_rare(a, kFB, b, dr.j | (kModeQ << 8));
    return;
  }
  int token = -1;
  bool cert = false;
  if (Sr.hi > 0.0f) {
    const RowPtrs<E> rp = row_ptrs<E>(a, b);
    AccEntries<E> ae;
    ae.tq = reinterpret_cast<const uint4*>(rp.tgt + size_t(dr.j) * a.V);
    ae.tp = dr.pair ? reinterpret_cast<const uint4*>(rp.drf + size_t(dr.j) * a.V) : nullptr;
    ae.pair = dr.pair;
    ae.tauq = thr_of(a, b, true, dr.j);
    ae.taup = dr.pair ? thr_of(a, b, false, dr.j) : -INFINITY;
    ae.Chi = a.Chi;
    ae.Clo = a.Clo;
    ae.Kq = Kq;
    ae.Kp = Kp;
    ae.Iq = Iq;
    ae.Ip = Ip;
    ae.tab = L.tab2;
    token = search_draw<E>(a, b, ae, sl, df_mul_f(Sr, uK), Eb, cert, PlainUnits{&a, b});
  }
  const int fl = flags | (cert ? 0 : SPEC_ROW_UNCERTIFIED);
  if (token < 0 && lane == 0 && a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
  write_outputs(a, b, dr.j, token, fl, token < 0, d);
}

// Combines the per-warp partials of a finished task and stores them as the
// task's slice partials in the workspace.
__device__ void combine_task(const SampleArgs& a, const QTask& t, const uint8_t* slot) {
  const int lane = threadIdx.x & 31;
  float* o = task_part(a, is_piece(t), t.b, t.s);
  if (t.type == kP1 || t.type == kBS) {
    // a per-position first-stage task covers rows 2 aux and 2 aux + 1
    const bool sub = a.p1sub && t.type == kP1;
    const int R = sub ? 2 : 2 * a.K, nrows = (t.type == kP1) ? R : 1;
    if (sub) o += 8 * t.aux;
    const float* w = reinterpret_cast<const float*>(slot + 16);
    const int* wb = reinterpret_cast<const int*>(w + 2 * R * kCW);
    for (int r = lane; r < nrows; r += 32) {
      float M = -INFINITY;
      int bad = 0;
#pragma unroll
      for (int q = 0; q < kCW; ++q) {
        M = fmaxf(M, w[r * kCW + q]);
        bad |= wb[r * kCW + q];
      }
      const float Kc = offset_of(M, a.c);
      df S{0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kCW; ++q) {
        const float s = w[(R + r) * kCW + q];
        if (s != 0.0f)
          S = df_add_f(S, __fmul_rn(s, pow2i(__fsub_rn(offset_of(w[r * kCW + q], a.c), Kc))));
      }
      o[4 * r] = M;
      o[4 * r + 1] = S.hi;
      o[4 * r + 2] = S.lo;
      o[4 * r + 3] = __int_as_float(bad);
    }
  } else if (lane == 0) {
    if (t.type == kSW) {
      const df* wd = reinterpret_cast<const df*>(slot + 16);
      const float* w = reinterpret_cast<const float*>(wd + kCW);
      df acc{0.f, 0.f};
      float aq = 0.f, ap = 0.f;
      for (int q = 0; q < kCW; ++q) {
        acc = df_add(acc, wd[q]);
        aq += w[q];
        ap += w[kCW + q];
      }
      o[0] = acc.hi;
      o[1] = acc.lo;
      o[2] = aq;
      o[3] = ap;
    } else if (t.type == kFA || t.type == kAR) {
      const df* w = reinterpret_cast<const df*>(slot + 16);
      df s0{0.f, 0.f}, s1{0.f, 0.f};
      for (int q = 0; q < kCW; ++q) {
        s0 = df_add(s0, w[q]);
        s1 = df_add(s1, w[kCW + q]);
      }
      o[0] = s0.hi;
      o[1] = s0.lo;
      o[2] = s1.hi;
      o[3] = s1.lo;
    } else if (t.type == kFR || t.type == kFD) {
      const df* w = reinterpret_cast<const df*>(slot + 16);
      df x[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
      for (int q = 0; q < kCW; ++q)
#pragma unroll
        for (int c = 0; c < 4; ++c) x[c] = df_add(x[c], w[c * kCW + q]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        o[2 * c] = x[c].hi;
        o[2 * c + 1] = x[c].lo;
      }
    } else {  // kFB
      const df* w = reinterpret_cast<const df*>(slot + 16);
      const float* f = reinterpret_cast<const float*>(w + kCW);
      df acc{0.f, 0.f};
      float qs = 0.f, ps = 0.f;
      for (int q = 0; q < kCW; ++q) {
        acc = df_add(acc, w[q]);
        qs += f[q];
        ps += f[kCW + q];
      }
      o[0] = acc.hi;
      o[1] = acc.lo;
      o[2] = qs;
      o[3] = ps;
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ consumers
// Each returns false on a timeout; `it` advances past the task's stages.

template <class E>
__device__ bool consume_stats(const SampleArgs& a, const Smem& L, uint32_t& it, uint8_t* slot,
                              const QTask& t) {
  const int tid = threadIdx.x;
  // rows per task: 2K (P1), 2 (P1 per position aux, small batches), 1 (BS)
  const bool sub = a.p1sub && t.type == kP1;
  const int R = sub ? 2 : 2 * a.K;
  const int pos0 = sub ? t.aux : 0;
  StatOp<E> op;
  op.c = a.c;
  op.tau = -INFINITY;
  op.begin();
  // P1 rows: target i = 2i, draft i = 2i + 1; BS: target row K
  auto tau_of = [&](int r) {
    return (t.type == kBS) ? thr_of(a, t.b, true, a.K)
                           : thr_of(a, t.b, (r & 1) == 0, pos0 + (r >> 1));
  };
  for (;;) {
    const ChunkMeta m = L.ring.meta[it % kStages];
    const uint4* buf = stage_data(L.ring, it);
    const int cnt = m.c1 - m.c0;
    if (E::kMask) op.tau = tau_of(m.r);
    op.chunk(buf, cnt, tid);
    release_stage(L.ring, it);
    if (m.last_k) {
      op.end_row(slot, R, m.r);
      op.begin();
    }
    ++it;
    if (m.last) return true;
    if (!wait_stage(L.ring, it)) return false;
  }
}

// Unit sums of one stage: vs[k] is this lane's vector (pair) sum of unit
// warp + kCons / 32 * k of the stage; the transposed warp reduction leaves
// unit k's sum on lanes (32 / N) k .. (32 / N) (k + 1) - 1.
// Returns the unit sum on the first lane of each unit's group, 0 elsewhere,
// so that the warp's sum of the returned values counts every unit once.
template <int N>
__device__ __forceinline__ float store_units(float (&vs)[N], float2* units, int u0, int cnt) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = lane / (32 / N);
  const float us = warp_sum_slots<N>(vs);
  const int i0 = warp * 32 + k * kCons;
  const bool mine = lane % (32 / N) == 0 && i0 < cnt;
  if (mine) units[u0 + i0 / 32] = make_float2(us, 0.f);
  return mine ? us : 0.0f;
}

template <class E>
__device__ bool consume_sw(const SampleArgs& a, const Smem& L, uint32_t& it, uint8_t* slot,
                           const QTask& t) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DrawRows dr = draw_rows(a.K, t.aux);
  const RowState* st = row_state(a, t.b);
  FastEntries<E> fe;
  fe.tq = nullptr;  // the sweep reads the ring stages
  fe.tp = nullptr;
  fe.pair = dr.pair;
  fe.c = a.c;
  fe.tauq = thr_of(a, t.b, true, dr.j);
  fe.taup = dr.pair ? thr_of(a, t.b, false, dr.j) : -INFINITY;
  fe.Kq = __ldcg(&st->Kq);
  fe.Rq = __ldcg(&st->Rq);
  fe.Kp = dr.pair ? __ldcg(&st->Kp) : 0.f;
  fe.Rp = dr.pair ? __ldcg(&st->Rp) : 0.f;
  fe.absx = (t.aux & kRawBit) != 0;
  int v0, v1;
  slice_range(a.nvec, a.S, t.s, v0, v1);
  // the slice total is the pair-arithmetic sum of its unit sums, so slice and
  // unit prefixes come from one summation tree (depth 3 + 5 per term)
  df acc{0.f, 0.f};
  float Aq = 0.f, Ap = 0.f;
  float2* units = a.ws.units(t.b, t.s);
  bool ok = true;
  for (;;) {
    const ChunkMeta m = L.ring.meta[it % kStages];
    const uint4* bq = stage_data(L.ring, it);
    const int cnt = m.c1 - m.c0;
    const int u0 = (m.c0 - v0) / 32;
    if (dr.pair) {
      // a stage holds the same vectors of both rows, q first, then p
      constexpr int kPer = kChunk / 32 / kCons;
      const uint4* bp = bq + kChunk / 32;
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
      acc = df_add_f(acc, store_units<kPer>(vs, units, u0, cnt));
    } else {
      constexpr int kPer = kChunk / 16 / kCons;
      float vs[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = warp * 32 + k * kCons + lane;
        vs[k] = 0.f;
        if (i < cnt) {
          float r[E::kVec];
          vs[k] = fe.run(bq[i], bq[i], r, Aq, Ap);
        }
      }
      acc = df_add_f(acc, store_units<kPer>(vs, units, u0, cnt));
    }
    release_stage(L.ring, it);
    ++it;
    if (m.last) break;
    if (!wait_stage(L.ring, it)) {
      ok = false;
      break;
    }
  }
  acc = df_warp_sum(acc);
  Aq = warp_sum_f(Aq);
  Ap = warp_sum_f(Ap);
  if (lane == 0) {
    df* wd = reinterpret_cast<df*>(slot + 16);
    float* w = reinterpret_cast<float*>(wd + kCW);
    wd[warp] = acc;
    w[warp] = Aq;
    w[kCW + warp] = Ap;
  }
  return ok;
}

// FA / AR: double-float sums of the task's rows (row 0 with offset K0, row 1
// with K1).
template <class E>
__device__ bool consume_rowsums(const SampleArgs& a, const Smem& L, uint32_t& it, uint8_t* slot,
                                const QTask& t) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const RowState* st = row_state(a, t.b);
  float K0, K1;
  if (t.type == kAR) {
    K0 = __ldcg(&st->rK[2 * (t.aux & 0xff)]);
    K1 = __ldcg(&st->rK[2 * (t.aux & 0xff) + 1]);
  } else {
    K0 = __ldcg(&st->Kq);
    K1 = draw_rows(a.K, t.aux).pair ? __ldcg(&st->Kp) : 0.f;
  }
  // rows: AR target / draft i, FA target / draft j
  const int ri = (t.type == kAR) ? (t.aux & 0xff) : draw_rows(a.K, t.aux).j;
  const bool two = (t.type == kAR) || draw_rows(a.K, t.aux).pair;  // draft row ri < K exists
  const float tau0 = thr_of(a, t.b, true, ri);
  const float tau1 = two ? thr_of(a, t.b, false, ri) : -INFINITY;
  df s0{0.f, 0.f}, s1{0.f, 0.f};
  bool ok = true;
  for (;;) {
    const ChunkMeta m = L.ring.meta[it % kStages];
    const uint4* buf = stage_data(L.ring, it);
    const float Kr = (m.r == 0) ? K0 : K1;
    const float tau = (m.r == 0) ? tau0 : tau1;
    df acc{0.f, 0.f};
    for (int i = tid; i < m.c1 - m.c0; i += kCons) {
      float z[E::kVec];
      E::unpack(buf[i], z);
      if (E::kMask) mask_vals(z, tau);
#pragma unroll
      for (int k = 0; k < E::kVec; ++k)
        acc = df_add(acc, acc_elem(z[k], a.Chi, a.Clo, Kr, L.tab2));
    }
    if (m.r == 0) s0 = df_add(s0, acc);
    else s1 = df_add(s1, acc);
    release_stage(L.ring, it);
    ++it;
    if (m.last) break;
    if (!wait_stage(L.ring, it)) {
      ok = false;
      break;
    }
  }
  s0 = df_warp_sum(s0);
  s1 = df_warp_sum(s1);
  if (lane == 0) {
    df* w = reinterpret_cast<df*>(slot + 16);
    w[warp] = s0;
    w[kCW + warp] = s1;
  }
  return ok;
}

// FB: double-float residual, unit sums and sums of q and p.
template <class E>
__device__ bool consume_fb(const SampleArgs& a, const Smem& L, uint32_t& it, uint8_t* slot,
                           const QTask& t) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DrawRows dr = draw_rows(a.K, t.aux);
  const RowState* st = row_state(a, t.b);
  AccEntries<E> ae;
  ae.tq = nullptr;  // the sweep reads the ring stages
  ae.tp = nullptr;
  ae.pair = dr.pair;
  ae.tauq = thr_of(a, t.b, true, dr.j);
  ae.taup = dr.pair ? thr_of(a, t.b, false, dr.j) : -INFINITY;
  ae.Chi = a.Chi;
  ae.Clo = a.Clo;
  ae.Kq = __ldcg(&st->Kq);
  ae.Kp = dr.pair ? __ldcg(&st->Kp) : 0.f;
  ae.Iq = df{__ldcg(&st->Iq_hi), __ldcg(&st->Iq_lo)};
  ae.Ip = dr.pair ? df{__ldcg(&st->Ip_hi), __ldcg(&st->Ip_lo)} : df{0.f, 0.f};
  ae.tab = L.tab2;
  int v0, v1, ps, pv0;
  task_range(a, is_piece(t), t.s, v0, v1, ps, pv0);
  df acc{0.f, 0.f};
  float Q = 0.f, P = 0.f;
  float2* units = a.ws.units(t.b, ps);  // the enclosing slice's unit sums
  bool ok = true;
  for (;;) {
    const ChunkMeta m = L.ring.meta[it % kStages];
    const uint4* bq = stage_data(L.ring, it);
    const uint4* bp = dr.pair ? bq + kChunk / 32 : bq;
    const int cnt = m.c1 - m.c0;
    for (int i0 = warp * 32; i0 < cnt; i0 += kCons) {
      const int i = i0 + lane;
      df vs{0.f, 0.f};
      if (i < cnt) {
        df r[E::kVec];
        vs = ae.run(bq[i], bp[i], r, Q, P);
      }
      const df us = df_warp_sum(vs);
      if (lane == 0) {
        units[(m.c0 - pv0 + i0) / 32] = make_float2(us.hi, us.lo);
        acc = df_add(acc, us);
      }
    }
    release_stage(L.ring, it);
    ++it;
    if (m.last) break;
    if (!wait_stage(L.ring, it)) {
      ok = false;
      break;
    }
  }
  acc = df_warp_sum(acc);
  Q = warp_sum_f(Q);
  P = warp_sum_f(P);
  if (lane == 0) {
    df* w = reinterpret_cast<df*>(slot + 16);
    w[warp] = acc;
    float* f = reinterpret_cast<float*>(w + kCW);
    f[warp] = Q;
    f[kCW + warp] = P;
  }
  return ok;
}

// Packed pair accumulation: (H, Lo) += (s, e) for two independent sums at
// once (halves of the f32x2 registers), TwoSum on the high parts, the errors
// and the low parts summed in Lo. With n additions the result is within
// 2 n^2 u^2 of the exact sum (relative), far below the exponentials' error.
__device__ __forceinline__ void acc2(uint64_t& H, uint64_t& Lo, uint64_t sh, uint64_t sl) {
  const uint64_t S = f2_add(H, sh);
  const uint64_t bb = f2_sub(S, H);
  const uint64_t err = f2_add(f2_sub(H, f2_sub(S, bb)), f2_sub(sh, bb));
  Lo = f2_add(Lo, f2_add(err, sl));
  H = S;
}

// Pair sum (as df_add) of two packed pairs, half by half.
__device__ __forceinline__ void df_add2(uint64_t& H, uint64_t& Lo, uint64_t yh, uint64_t yl) {
  const uint64_t s = f2_add(H, yh);
  const uint64_t bb = f2_sub(s, H);
  const uint64_t err = f2_add(f2_sub(H, f2_sub(s, bb)), f2_sub(yh, bb));
  const uint64_t e = f2_add(err, f2_add(Lo, yl));
  H = f2_add(s, e);
  Lo = f2_sub(e, f2_sub(H, s));
}

// Warp sum of two pairs at once (df_warp_sum of each half); every lane ends
// with the totals.
__device__ __forceinline__ void df_warp_sum2(uint64_t& H, uint64_t& Lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t yh = __shfl_xor_sync(0xffffffffu, H, o);
    const uint64_t yl = __shfl_xor_sync(0xffffffffu, Lo, o);
    df_add2(H, Lo, yh, yl);
  }
}

// FR: one pass over the draw's rows (see the header) with the lighter
// exponential (lite_exp2x2, relative error < kLiteExpRelErr) on packed pairs;
// FD (kDf): the same pass with the double-float exponential (df_exp2,
// relative error < 4e-13), for the rows FR leaves undecided.
// Per unit the pair sums of e_q and e_p over the tokens with a certainly
// positive residual; per task the row sums and the unit sums' totals;
// tokens inside the sign test's margin go to the row's list. Each term is
// first normalised to a pair (s, e) with |e| <= u |s| (FastTwoSum), so the
// accumulations keep the error bound of acc2.
template <class E, bool kDf>
__device__ bool consume_fr(const SampleArgs& a, const Smem& L, uint32_t& it, uint8_t* slot,
                           const QTask& t) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DrawRows dr = draw_rows(a.K, t.aux);
  RowState* st = row_state(a, t.b);
  const float Kq = __ldcg(&st->Kq), Kp = dr.pair ? __ldcg(&st->Kp) : 0.f;
  const float Rq = __ldcg(&st->Rq), Rp = dr.pair ? __ldcg(&st->Rp) : 0.f;
  const float up1 = 1.0f + (dr.pair ? __ldcg(&st->amb_delta) : 0.f);
  const float tauq = thr_of(a, t.b, true, dr.j);
  const float taup = dr.pair ? thr_of(a, t.b, false, dr.j) : -INFINITY;
  const LiteConsts LC = lite_consts(a.Chi, a.Clo);
  const LiteRow Lq = lite_row(Kq, a.Chi);
  const LiteRow Lp = dr.pair ? lite_row(Kp, a.Chi) : Lq;
  const uint64_t r2 = f2_pack(Rq, Rp);
  int v0, v1, ps, pv0;
  task_range(a, is_piece(t), t.s, v0, v1, ps, pv0);
  float4* units = reinterpret_cast<float4*>(a.ws.units(t.b, ps));
  const uint64_t zero2 = f2_pack(0.f, 0.f);
  uint64_t Th = zero2, Tl = zero2;  // (Tq, Tp) partial row sums of this thread
  df Aq{0.f, 0.f}, Ap{0.f, 0.f};
  bool ok = true;
  for (;;) {
    const ChunkMeta m = L.ring.meta[it % kStages];
    const uint4* bq = stage_data(L.ring, it);
    const uint4* bp = dr.pair ? bq + kChunk / 32 : bq;
    const int cnt = m.c1 - m.c0;
    for (int i0 = warp * 32; i0 < cnt; i0 += kCons) {
      const int i = i0 + lane;
      uint64_t Vh = zero2, Vl = zero2;  // this lane's (q, p) unit partials
      if (i < cnt) {
        float zq[E::kVec], zp[E::kVec];
        E::unpack(bq[i], zq);
        if (dr.pair) E::unpack(bp[i], zp);
        if (E::kMask) {
          mask_vals(zq, tauq);
          if (dr.pair) mask_vals(zp, taup);
        }
        if (dr.pair) {
#pragma unroll
          for (int k = 0; k < E::kVec; ++k) {
            df eq, ep;
            if (kDf) {
              eq = acc_elem(zq[k], a.Chi, a.Clo, Kq, L.tab2);
              ep = acc_elem(zp[k], a.Chi, a.Clo, Kp, L.tab2);
            } else {
              lite_exp2x2(zq[k], zp[k], Lq, Lp, LC, L.tab2, eq, ep);
            }
            const uint64_t h = f2_pack(eq.hi, ep.hi), l = f2_pack(eq.lo, ep.lo);
            const uint64_t sh = f2_add(h, l);
            const uint64_t sl = f2_sub(l, f2_sub(sh, h));
            acc2(Th, Tl, sh, sl);
            float x, y;
            f2_unpack(f2_mul(sh, r2), x, y);
            const bool pos = x > __fmul_rn(y, up1);
            if (pos) {
              acc2(Vh, Vl, sh, sl);
            } else if (!(__fmul_rn(x, up1) <= y)) {
              const int slot_i = atomicAdd(&st->namb, 1);
              if (slot_i < kAmbCap) {
                float qh, ph, ql, pl;
                f2_unpack(sh, qh, ph);
                f2_unpack(sl, ql, pl);
                AmbEntry e;
                e.v = (m.c0 + i) * E::kVec + k;
                e.pad = 0;
                e.qh = qh;
                e.ql = ql;
                e.ph = ph;
                e.pl = pl;
                st->amb[slot_i] = e;
              }
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < E::kVec; k += 2) {
            df e0, e1;
            if (kDf) {
              e0 = acc_elem(zq[k], a.Chi, a.Clo, Kq, L.tab2);
              e1 = acc_elem(zq[k + 1], a.Chi, a.Clo, Kq, L.tab2);
            } else {
              lite_exp2x2(zq[k], zq[k + 1], Lq, Lq, LC, L.tab2, e0, e1);
            }
            const uint64_t h = f2_pack(e0.hi, e1.hi), l = f2_pack(e0.lo, e1.lo);
            const uint64_t sh = f2_add(h, l);
            const uint64_t sl = f2_sub(l, f2_sub(sh, h));
            acc2(Th, Tl, sh, sl);
            acc2(Vh, Vl, sh, sl);
          }
        }
      }
      if (!dr.pair) {
        // both halves hold q terms: fold them into the first half
        float h0, h1, l0, l1;
        f2_unpack(Vh, h0, h1);
        f2_unpack(Vl, l0, l1);
        const df v = df_add(df{h0, l0}, df{h1, l1});
        Vh = f2_pack(v.hi, 0.f);
        Vl = f2_pack(v.lo, 0.f);
      }
      df_warp_sum2(Vh, Vl);
      if (lane == 0) {
        float uqh, uph, uql, upl;
        f2_unpack(Vh, uqh, uph);
        f2_unpack(Vl, uql, upl);
        units[(m.c0 - pv0 + i0) / 32] = make_float4(uqh, uql, uph, upl);
        Aq = df_add(Aq, df{uqh, uql});
        Ap = df_add(Ap, df{uph, upl});
      }
    }
    release_stage(L.ring, it);
    ++it;
    if (m.last) break;
    if (!wait_stage(L.ring, it)) {
      ok = false;
      break;
    }
  }
  if (!dr.pair) {
    float h0, h1, l0, l1;
    f2_unpack(Th, h0, h1);
    f2_unpack(Tl, l0, l1);
    const df v = df_add(df{h0, l0}, df{h1, l1});
    Th = f2_pack(v.hi, 0.f);
    Tl = f2_pack(v.lo, 0.f);
  }
  df_warp_sum2(Th, Tl);
  if (lane == 0) {
    float tqh, tph, tql, tpl;
    f2_unpack(Th, tqh, tph);
    f2_unpack(Tl, tql, tpl);
    df* w = reinterpret_cast<df*>(slot + 16);
    w[warp] = df{tqh, tql};
    w[kCW + warp] = df{tph, tpl};
    w[2 * kCW + warp] = Aq;
    w[3 * kCW + warp] = Ap;
  }
  return ok;
}

// FR / FD complete: accurate normalisers, the ambiguous tokens decided
// exactly, residual unit sums and the certified search; a draw FR leaves
// undecided goes to FD, a list overflow (or a degenerate row) to FA / FB.
template <class E, bool kDf>
__device__ void finish_fr(const SampleArgs& a, const Smem& L, int b, int aux) {
  const int lane = threadIdx.x & 31;
  RowState* st = row_state(a, b);
  const DrawRows dr = draw_rows(a.K, aux);
  const bool pieces = aux & kPieceBit;
  const int np = pieces ? a.R : a.S;
  const int d = load_tokens(a, b);
  const int flags = __ldcg(&st->flags);
  const float Kq = __ldcg(&st->Kq), Kp = dr.pair ? __ldcg(&st->Kp) : 0.f;
  const float uK = a.uniforms[size_t(b) * (a.K + 1) + a.K];
  // lanes hold parts lane and lane + 32: (Tq, Tp, Aq, Ap)
  df tq[2], tp[2], aq[2], ap[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    tq[h] = tp[h] = aq[h] = ap[h] = df{0.f, 0.f};
    const int sidx = lane + 32 * h;
    if (sidx < np) {
      const float4* w = reinterpret_cast<const float4*>(task_part(a, pieces, b, sidx));
      const float4 v0 = __ldcg(w), v1 = __ldcg(w + 1);
      tq[h] = df{v0.x, v0.y};
      tp[h] = df{v0.z, v0.w};
      aq[h] = df{v1.x, v1.y};
      ap[h] = df{v1.z, v1.w};
    }
  }
  const df Sq = df_warp_sum(df_add(tq[0], tq[1]));
  const df Sp = dr.pair ? df_warp_sum(df_add(tp[0], tp[1])) : df{0.f, 0.f};
  const int namb = dr.pair ? __ldcg(&st->namb) : 0;
  if (!(Sq.hi > 0.0f) || (dr.pair && !(Sp.hi > 0.0f)) || namb > kAmbCap) {
    // list overflow (or a degenerate row): the two-pass FA / FB path
    enqueue_rare(a, kFA, b, aux & ~kPieceBit);
    return;
  }
  const df Iq = df_recip(Sq), Ip = dr.pair ? df_recip(Sp) : df{0.f, 0.f};
  // ambiguous tokens: residual e_q/S_q - e_p/S_p in pair arithmetic, kept if positive
  int av = -1;
  df ad{0.f, 0.f};
  if (lane < namb) {
    const AmbEntry e = st->amb[lane];
    av = e.v;
    ad = df_sub(df_mul(df{e.qh, e.ql}, Iq), df_mul(df{e.ph, e.pl}, Ip));
    if (!(ad.hi > 0.0f)) ad = df{0.f, 0.f};
  }
  const int apart = lane < namb ? part_of_token(a, pieces, av) : -1;
  // residual of each part
  DrawSlices sl;
  sl.pieces = pieces;
  sl.n = np;
  df xr[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    xr[h] = df_mul(aq[h], Iq);
    if (dr.pair) xr[h] = df_sub(xr[h], df_mul(ap[h], Ip));
    for (int e = 0; e < namb; ++e) {
      const int pe = __shfl_sync(0xffffffffu, apart, e);
      const df de = df_shfl(ad, e);
      if (pe == lane + 32 * h) xr[h] = df_add(xr[h], de);
    }
  }
  sl.xa = xr[0];
  sl.xb = xr[1];
  sl.total = df_warp_sum(df_add(xr[0], xr[1]));
  sl.f2 = sl.f3 = 0.f;
  const df Sr = sl.total;
  if (!(Sr.hi > 0.0f) && dr.pair) {
    // zero residual mass: the draw uses q_j itself
    if (lane == 0) st->flags = flags | SPEC_ROW_ZERO_RESIDUAL;  // (a q-only pass keeps no list of tokens)
    enqueue_rare(a, kDf ? kFD : kFR, b, dr.j | (kModeQ << 8));
    return;
  }
  // Error bound: per token, relative error below kFrRho for e_q / S_q and
  // e_p / S_p (FR's exponential in the term and in the normaliser, the pair
  // sums and the reciprocal), whatever the order of the pair-arithmetic sums
  // and products; summed with weights q and p (total 1 each, margin 10%). The
  // walk of the final unit recomputes its terms the same way. A token whose
  // sign is undecidable within that error moves by at most its own error.
  const float rho = kDf ? fmaxf(acc_rho(Kq), acc_rho(Kp)) : kFrRho;
  const float Eb = 1.1f * rho * (dr.pair ? 2.0f : 1.0f) + 1e-14f * Sr.hi + 1e-36f;
  int token = -1;
  bool cert = false;
  {
    const RowPtrs<E> rp = row_ptrs<E>(a, b);
    FrUnits fu{&a, b, namb, av, dr.pair, Iq, Ip, ad};
    if (kDf) {
      AccEntries<E> ae;
      ae.tq = reinterpret_cast<const uint4*>(rp.tgt + size_t(dr.j) * a.V);
      ae.tp = dr.pair ? reinterpret_cast<const uint4*>(rp.drf + size_t(dr.j) * a.V) : nullptr;
      ae.pair = dr.pair;
      ae.tauq = thr_of(a, b, true, dr.j);
      ae.taup = dr.pair ? thr_of(a, b, false, dr.j) : -INFINITY;
      ae.Chi = a.Chi;
      ae.Clo = a.Clo;
      ae.Kq = Kq;
      ae.Kp = Kp;
      ae.Iq = Iq;
      ae.Ip = Ip;
      ae.tab = L.tab2;
      token = search_draw<E>(a, b, ae, sl, df_mul_f(Sr, uK), Eb, cert, fu);
    } else {
      LiteEntries<E> le;
      le.tq = reinterpret_cast<const uint4*>(rp.tgt + size_t(dr.j) * a.V);
      le.tp = dr.pair ? reinterpret_cast<const uint4*>(rp.drf + size_t(dr.j) * a.V) : nullptr;
      le.pair = dr.pair;
      le.tauq = thr_of(a, b, true, dr.j);
      le.taup = dr.pair ? thr_of(a, b, false, dr.j) : -INFINITY;
      le.LC = lite_consts(a.Chi, a.Clo);
      le.Lq = lite_row(Kq, a.Chi);
      le.Lp = dr.pair ? lite_row(Kp, a.Chi) : le.Lq;
      le.Iq = Iq;
      le.Ip = Ip;
      le.tab = L.tab2;
      token = search_draw<E>(a, b, le, sl, df_mul_f(Sr, uK), Eb, cert, fu);
    }
  }
  if (kDf || (token >= 0 && cert)) {
    // FD's bound is the final word: a draw even FD leaves undecided is flagged
    const int fl = flags | (cert ? 0 : SPEC_ROW_UNCERTIFIED);
    if (token < 0 && lane == 0 && a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
    write_outputs(a, b, dr.j, token, fl, token < 0, d);
    return;
  }
  // not settled within FR's bound: one double-float pass of the same kind
  // (FD), which rebuilds the list of undecided tokens from its own values
  if (lane == 0) {
    st->flags = flags | SPEC_ROW_SAMPLE_REFINED;
    st->namb = 0;
  }
  enqueue_rare(a, kFD, b, aux & ~kPieceBit);
}

// Logit rows a task streams: their number, whether they are read element by
// element in pairs, and (task_row) the base pointer of row r.
__device__ inline int task_nrows(const SampleArgs& a, const QTask& t, bool& paired) {
  paired = false;
  if (t.type == kP1) return a.p1sub ? 2 : 2 * a.K;
  if (t.type == kBS) return 1;
  if (t.type == kAR) return 2;
  const DrawRows dr = draw_rows(a.K, t.aux);
  paired = dr.pair && t.type != kFA;
  return dr.pair ? 2 : 1;
}
template <class E>
__device__ inline const char* task_row(const SampleArgs& a, const QTask& t, int r) {
  const RowPtrs<E> rp = row_ptrs<E>(a, t.b);
  int i;
  bool tgt = true;
  if (t.type == kP1) {  // target i = row 2i, draft i = row 2i + 1
    i = (a.p1sub ? t.aux : 0) + (r >> 1);
    tgt = (r & 1) == 0;
  } else if (t.type == kBS) {
    i = a.K;
  } else if (t.type == kAR) {
    i = t.aux & 0xff;
    tgt = r == 0;
  } else {
    i = draw_rows(a.K, t.aux).j;
    tgt = r == 0;
  }
  return reinterpret_cast<const char*>(tgt ? rp.tgt + size_t(i) * a.V : rp.drf + size_t(i) * a.V);
}

// ------------------------------------------------------------------ kernel
template <class E>
__global__ void __launch_bounds__(kThreads, 2) verify_sample_kernel(const SampleArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int K = a.K;
  const Smem L = make_smem(smem_raw, 2 * K);
  ring_init(L.ring);
  handoff_init(L.ho);
  for (int i = threadIdx.x; i < 256; i += kThreads)
    L.tab2[i] = make_float2(kExp2Tab.hi[i], kExp2Tab.lo[i]);
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
        if (!fx.next(a.ws, kP1, t)) {
          if (!producer_idle(a.ws, !fx.first_left, idle_t0)) break;
          continue;
        }
        idle_t0 = 0;
        int v0, v1, ps, pv0;
        task_range(a, is_piece(t), t.s, v0, v1, ps, pv0);
        bool paired;
        const int nrows = task_nrows(a, t, paired);
        auto row = [&](int r) { return task_row<E>(a, t, r); };
        auto prefetch = [&]() { fx.prepare(a.ws); };
        if (!produce_task(L.ring, it, nt, t, row, nrows, paired, v0, v1, prefetch)) break;
      }
      produce_end(L.ring, it);
    }
  } else if (warp == kFinWarp) {
    // ------------------------------------------------ finisher
    finisher_loop(
        a.ws, L.ho, L.ring.abort,
        [&](const QTask& t, const uint8_t* slot) { combine_task(a, t, slot); },
        [&](const QTask& t) {
          switch (t.type) {
            case kP1:
              finish_p1<E>(a, L, t.b);
              break;
            case kAR:
              finish_ar<E>(a, L, t.b, t.aux);
              break;
            case kBS:
              finish_bs(a, L, t.b);
              break;
            case kSW:
              finish_sw<E>(a, t.b, t.aux);
              break;
            case kFA:
              finish_fa(a, t.b, t.aux);
              break;
            case kFR:
              finish_fr<E, false>(a, L, t.b, t.aux);
              break;
            case kFD:
              finish_fr<E, true>(a, L, t.b, t.aux);
              break;
            default:
              finish_fb<E>(a, L, t.b, t.aux);
              break;
          }
        },
        [&](const QTask& t) {
          return is_piece(t) ? a.R : (t.type == kP1 && a.p1sub) ? a.S * a.K : a.S;
        });
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
      bool ok;
      if (t.type == kP1 || t.type == kBS) ok = consume_stats<E>(a, L, it, slot, t);
      else if (t.type == kSW) ok = consume_sw<E>(a, L, it, slot, t);
      else if (t.type == kFA || t.type == kAR) ok = consume_rowsums<E>(a, L, it, slot, t);
      else if (t.type == kFR) ok = consume_fr<E, false>(a, L, it, slot, t);
      else if (t.type == kFD) ok = consume_fr<E, true>(a, L, it, slot, t);
      else ok = consume_fb<E>(a, L, it, slot, t);
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

}  // namespace

// ------------------------------------------------------------------ host side
namespace {

// Refinement pieces per slice: up to 3 (measured best on the bench workload
// among 1, 2, 3, 4 and 8; at most kMaxSlices per row), no more than the
// 32-vector units of the smallest slice.
int pieces_per_slice(int nvec, int S) {
  int m = kMaxSlices / S;
  if (m > 3) m = 3;
  const int min_units = (nvec / S + 31) / 32;
  if (m > min_units) m = min_units;
  return m < 1 ? 1 : m;
}

WsLayout sample_layout(int B, int K, int V, int dtype) {
  const int kvec = (dtype == SPEC_BF16) ? 8 : 4;
  const int nvec = V / kvec;
  const bool small = small_batch(B, small_batch_knob(), kSampleSmallBatch);
  const int S = slices_for(nvec, B, small, kSampleTasks);
  const int M = pieces_per_slice(nvec, S);
  const int maxslice = (nvec + S - 1) / S;
  // unit slots (float2) per slice: FR keeps two pairs per unit (float4)
  const int ustride = 2 * ((maxslice + 31) / 32) + 2;
  int part = (8 * K > 8) ? 8 * K : 8;  // P1: 4 floats for each of the 2K rows; FR: 8
  if (part < 8 * M) part = 8 * M;      // a row's S blocks hold its R = S M piece partials
  // queued tasks per row: BS, SW (S each); FR and FD twice each (zero
  // residual), FA, FB twice, AR up to K times (R = S M each)
  WsLayout w = ws_layout(B, S, part, ustride, (8 + K) * M, int(sizeof(RowState)));
  // small batches: one first-stage task per (slice, position) when that
  // still fits one task per persistent CTA
  if (small && B * S * K <= kOneWave) w.kp = K;
  return w;
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
  a.M = pieces_per_slice(a.nvec, a.S);
  a.R = a.S * a.M;
  a.ws.base = static_cast<uint8_t*>(s.workspace);
  a.ws.L = wl;
  a.p1sub = wl.kp > 1 ? 1 : 0;
  const int knob = small_batch_knob();
  a.direct_fr = knob >= 0 ? knob : (s.B >= 4 && s.B <= kSampleSmallBatch) ? 1 : 0;
  set_test_knobs(a.ws);
  const double C = 1.4426950408889634073599246810018921 / double(s.temperature);  // log2(e)/T
  a.c = float(C);
  a.Chi = float(C);
  a.Clo = float(C - double(a.Chi));
  // fp32 additions a row sum goes through before the double-float combine:
  // per thread at most `run` (vectors of a row slice per thread + 2), the
  // 8-term tree of a vector (3) and the warp tree (5)
  const int maxslice = (a.nvec + a.S - 1) / a.S;
  const int run = maxslice / kCons + 2;
  a.bd.ex2 = float(kEx2RelErrBound);
  a.bd.gamma1 = float((3.0 + 5.0 + run) * 5.9604644775390625e-8 * 1.01);
  a.bd.xbar = float(std::log2(double(s.V)) + 2.0);
  a.out_tokens = s.out_tokens;
  a.out_n = s.out_n;
  a.err = s.err;
  a.row_info = s.row_info;
  a.q_at_d = s.q_at_d;
  a.p_at_d = s.p_at_d;
  a.counters = s.counters;
  a.thr_t = s.thr_t;
  a.thr_d = s.thr_d;
  a.masked = (s.thr_t || s.thr_d) ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(s.stream);
  if (zero_workspace(s.workspace, wl.zero_bytes, st) != SPEC_OK) return SPEC_ECUDA;
  const size_t smem = sample_smem_bytes(2 * s.K);
  if (a.masked) {
    if (s.dtype == SPEC_BF16)
      return launch_dataflow(verify_sample_kernel<EM<EBf16, true>>, a, smem, st);
    return launch_dataflow(verify_sample_kernel<EM<EF32, true>>, a, smem, st);
  }
  if (s.dtype == SPEC_BF16) return launch_dataflow(verify_sample_kernel<EM<EBf16, false>>, a, smem, st);
  return launch_dataflow(verify_sample_kernel<EM<EF32, false>>, a, smem, st);
}

}  // namespace sv
