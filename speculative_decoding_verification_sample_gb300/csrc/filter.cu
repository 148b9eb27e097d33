// Top-k / top-p logit thresholds (spec_filter_thresholds).
//
// Method: "quickscale.ai - Quand et pourquoi utiliser le speculative
// decoding", section "Influence du sampling", names temperature, top-k and
// top-p as the sampling parameters that shape the verified distributions.
// Reading used (the pages give no definition): temperature, then top-k
// (every token whose logit is at least the k-th largest), then top-p on the
// renormalised top-k distribution (every token whose logit is at least the
// largest value t at which the tokens with logit >= t reach probability p).
// The result is one logit threshold per row; verification treats the tokens
// below it as logit -inf.
//
// GB300 mapping: one CTA per row, a radix selection on order-preserving
// integer keys of the logits (16 bits for bf16, 32 for fp32), 8 bits per
// level. Top-k needs only counts, so it is exact. Top-p needs probability
// mass: each token's mass 2^(z c - Kc) (c = log2(e)/T, Kc the row's integer
// offset) is rounded to a 64-bit fixed-point integer and summed with
// shared-memory integer atomics, which is exact and independent of the
// order. The fast pass takes the mass from the MUFU exp2 and certifies the
// final comparison against p with a proven bound on that mass's error; a row
// it cannot certify gets NaN, and the second launch recomputes exactly those
// rows with double-float exponentials (relative error < 1e-11).
// bf16 rows first take a two-pass kernel (filter_topk_bf16_kernel): the
// exact counts of the 256 keys below the row maximum give the k-th largest
// logit, top-p on the kept tokens follows from those bins' masses in fp64,
// and top-p alone from them plus the fp32 mass below the window, certified;
// the rows it cannot settle go to the kernels above.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/specverify.h"
#include "common.cuh"
#include "df.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace sv {
namespace {

constexpr int kFT = 256;      // threads per CTA, one row per CTA
constexpr int kFTAcc = 1024;  // the double-float rerun of the few uncertain rows
constexpr int kCand = 8;      // top-digit bins a one-pass top-p search may span

// Order-preserving keys: larger key <=> larger value (NaN excluded).
template <class E>
struct KeyOf;
template <>
struct KeyOf<EBf16> {
  static constexpr int kBits = 16;
  __device__ static __forceinline__ uint32_t key(float z) {
    const uint32_t b = __float_as_uint(z) >> 16;
    return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
  }
  __device__ static __forceinline__ float value(uint32_t k) {
    const uint32_t b = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
    return __uint_as_float(b << 16);
  }
};
template <>
struct KeyOf<EF32> {
  static constexpr int kBits = 32;
  __device__ static __forceinline__ uint32_t key(float z) {
    const uint32_t b = __float_as_uint(z);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  __device__ static __forceinline__ float value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
  }
};

struct FilterArgs {
  const void* logits;
  int R, V, nvec, top_k;
  float top_p, T, c, Chi, Clo, ex2, fixscale;
  int skip_done;  // general kernel after the bf16 top-k kernel: rows not NaN are done
  float* out;
  int32_t* err;
};

// Nonnegative float (below 2^62) to a fixed-point integer, within 1 of its
// value: the significand shifted by the exponent (plain integer operations,
// no conversion instruction).
__device__ __forceinline__ unsigned long long to_fixed(float f) {
  const uint32_t b = __float_as_uint(f);
  const int e = int(b >> 23) - 127;
  if (e < 0) return f >= 0.5f ? 1ull : 0ull;
  const unsigned long long m = (b & 0x7fffffu) | 0x800000u;
  return e >= 23 ? (m << (e - 23)) : (m >> (23 - e));
}

// Certification slack of one histogram bin's mass (fixed-point units): the
// relative error of each token's mass there is at most ex2 + ln2 u (2|x| + 2)
// with |x| <= xmax (argument and temperature-constant rounding; the part of
// the latter common to all tokens cancels in the ratio to the row total).
__device__ __forceinline__ double bin_err(unsigned long long m, float eps, float xmax) {
  if (m == 0) return 0.0;
  const float x = fminf(xmax, 200.0f);
  return double(m) * double(eps + kLn2f * kU * (2.0f * x + 2.0f)) * 1.02;
}

template <class E, bool kAcc>
__global__ void __launch_bounds__(kAcc ? kFTAcc : kFT) filter_kernel(const FilterArgs a) {
  using KO = KeyOf<E>;
  constexpr int NT = kAcc ? kFTAcc : kFT;
  constexpr int KB = KO::kBits, ND = KB / 8;
  __shared__ uint32_t hcnt[256];
  __shared__ unsigned long long hmass[256];
  __shared__ unsigned long long hbuck[256];
  __shared__ uint32_t s_u[NT / 32];
  __shared__ int s_i[NT / 32];
  __shared__ uint32_t s_need, s_digit;
  __shared__ unsigned long long s_A, s_mb, s_Z;
  __shared__ double s_EA, s_EZ;
  __shared__ unsigned long long s_red[NT / 32], s_ztot;
  __shared__ uint32_t s_floor, s_bl, s_bh, s_pre16;
  __shared__ int s_cand;
  __shared__ unsigned long long hwarp[NT / 32][256];  // per-warp level-0 masses
  __shared__ float s_th[kAcc ? 256 : 1], s_tl[kAcc ? 256 : 1];
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the accurate launch takes the uncertain rows only; so does the fast
  // launch after the bf16 top-k kernel (the rows it left)
  if ((kAcc || a.skip_done) && !isnan(a.out[row])) return;
  if (kAcc) {
    for (int i = tid; i < 256; i += NT) {
      s_th[i] = kExp2Tab.hi[i];
      s_tl[i] = kExp2Tab.lo[i];
    }
  }
  const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const char*>(a.logits) +
                                                   size_t(row) * size_t(a.V) * sizeof(typename E::T));
  const bool topk = a.top_k > 0 && a.top_k < a.V;
  const bool topp = a.top_p < 1.0f;
  auto sweep = [&](auto&& f) {
    for (int i = tid; i < a.nvec; i += NT) {
      float z[E::kVec];
      E::unpack(ldg_nc_v4(rp + i), z);
#pragma unroll
      for (int k = 0; k < E::kVec; ++k) f(z[k]);
    }
  };
  auto clear = [&]() {
    for (int i = tid; i < 256; i += NT) {
      hcnt[i] = 0;
      hmass[i] = 0;
      hbuck[i] = 0;
    }
  };
  // ---- pass 0: maximum key, NaN, top-k level-0 counts
  clear();
  __syncthreads();
  uint32_t mk = 0;
  int nan = 0;
  sweep([&](float z) {
    if (z != z) {
      nan = 1;
      return;
    }
    const uint32_t k = KO::key(z);
    mk = max(mk, k);
    if (topk || topp) atomicAdd(&hcnt[k >> (KB - 8)], 1u);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    nan |= __shfl_xor_sync(0xffffffffu, nan, o);
  }
  if (lane == 0) {
    s_u[warp] = mk;
    s_i[warp] = nan;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t m = 0;
    int n = 0;
    for (int w = 0; w < NT / 32; ++w) {
      m = max(m, s_u[w]);
      n |= s_i[w];
    }
    s_u[0] = m;
    s_i[0] = n;
  }
  __syncthreads();
  mk = s_u[0];
  if (s_i[0]) {  // NaN logits: every token filtered; the verification reports the row
    if (tid == 0) {
      a.out[row] = INFINITY;
      if (a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
    }
    return;
  }
  const float maxv = KO::value(mk);
  if (!(maxv > -INFINITY) || (!topk && !topp)) {
    if (tid == 0) a.out[row] = -INFINITY;
    return;
  }
  const float Kc = offset_of(maxv, a.c);
  if (topp && !(fabsf(Kc) < kMaxOffset)) {  // max * log2(e)/T out of range (or +inf)
    if (tid == 0) {
      a.out[row] = INFINITY;
      if (a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
    }
    return;
  }
  // fixed-point mass of one token (0 for -inf)
  auto mass = [&](float z) -> unsigned long long {
    if (kAcc) {
      const df p = two_prod(z, a.Chi);
      const float pl = __fmaf_rn(z, a.Clo, p.lo);
      const df s = two_sum(p.hi, -Kc);
      const df w = df_exp2(s.hi, __fadd_rn(s.lo, pl), s_th, s_tl);
      const float l = __fmul_rn(w.lo, a.fixscale);
      const unsigned long long h = to_fixed(__fmul_rn(w.hi, a.fixscale));
      const unsigned long long lm = to_fixed(fabsf(l));
      return l >= 0.0f ? h + lm : h - lm;
    }
    return to_fixed(__fmul_rn(ex2_approx(__fmaf_rn(z, a.c, -Kc)), a.fixscale));
  };
  const float eps = kAcc ? 2e-12f + 2.2e-14f * (fabsf(Kc) + 256.0f) : a.ex2;
  // |x| bound of the tokens in the key range starting at key k0
  auto xmax_from = [&](uint32_t k0) { return Kc - __fmul_rn(KO::value(k0), a.c) + 1.0f; };

  // ---- top-k: radix selection on counts
  uint32_t KA = 0;  // keep keys >= KA
  if (topk) {
    uint32_t pre = 0, need = uint32_t(a.top_k);
    for (int lvl = 0; lvl < ND; ++lvl) {
      const int sh = KB - 8 * (lvl + 1);  // shift of this level's digit
      if (lvl > 0) {
        __syncthreads();
        clear();
        __syncthreads();
        const bool last = lvl == ND - 1;
        sweep([&](float z) {
          const uint32_t k = KO::key(z);
          const uint32_t up = k >> (sh + 8);
          if (up == pre) atomicAdd(&hcnt[(k >> sh) & 255u], 1u);
          if (topp && last) {  // top-p level-0 masses, merged into this pass
            if (up > pre) {
              const unsigned long long q = mass(z);
              if (q) atomicAdd(&hmass[k >> (KB - 8)], q);
            } else if (up == pre) {
              const unsigned long long q = mass(z);
              if (q) atomicAdd(&hbuck[k & 255u], q);
            }
          }
        });
        __syncthreads();
      }
      if (tid == 0) {
        uint32_t cum = 0, d = 0;
        for (int b = 255; b >= 0; --b) {
          if (cum + hcnt[b] >= need) {
            d = uint32_t(b);
            break;
          }
          cum += hcnt[b];
        }
        s_digit = d;
        s_need = need - cum;
      }
      __syncthreads();
      pre = (pre << 8) | s_digit;
      need = s_need;
    }
    KA = pre;
  }
  float tau = topk ? KO::value(KA) : -INFINITY;

  // ---- top-p: radix selection on fixed-point masses of the keys >= KA
  if (topp) {
    __syncthreads();
    if (topk) {
      // the merged pass left the masses of keys above KA's last-level bucket
      // by top digit (hmass) and the bucket's masses by last digit (hbuck)
      if (tid == 0) {
        unsigned long long add = 0;
        for (int d = int(KA & 255u); d < 256; ++d) add += hbuck[d];
        hmass[KA >> (KB - 8)] += add;
        for (int d = 0; d < int(KA & 255u); ++d) hbuck[d] = 0;  // below KA: not kept
      }
    } else {
      // the row total Z, summed per thread (no atomics)
      unsigned long long zt = 0;
      sweep([&](float z) { zt += mass(z); });
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) zt += __shfl_xor_sync(0xffffffffu, zt, o);
      if (lane == 0) s_red[warp] = zt;
      __syncthreads();
      if (tid == 0) {
        unsigned long long Z = 0;
        for (int w = 0; w < NT / 32; ++w) Z += s_red[w];
        s_ztot = Z;
        // Candidate top-digit bins of t*: per bin, count x (mass of its
        // highest key) bounds the bin's mass from above and count x (mass of
        // its lowest key) from below; t*'s bin b* has mass(bins > b*) < p Z <=
        // mass(bins >= b*), so it lies in [bl, bh]: bh the highest bin whose
        // upper-bounded mass from the top reaches p Z, bl the lowest whose
        // lower-bounded mass strictly above stays below p Z.
        const double pZ = double(a.top_p) * double(Z);
        double ub = 0.0, lbab = 0.0, ez = 0.0, ea = 0.0;
        int bh = -1, bl = -1;
        for (int b = 255; b >= 0; --b) {
          const uint32_t k0 = uint32_t(b) << (KB - 8), k1 = k0 | ((1u << (KB - 8)) - 1u);
          const float zh = KO::value(k1), zl = KO::value(k0);
          const float wh = (zh == zh) ? ex2_approx(fminf(__fmaf_rn(zh, a.c, -Kc), 1.0f)) : 0.0f;
          const float wl = (zl == zl) ? ex2_approx(fminf(__fmaf_rn(zl, a.c, -Kc), 1.0f)) : 0.0f;
          const double n = double(hcnt[b]);
          const double mhi = n * (double(wh) * 1.01 * double(a.fixscale) + 1.0);
          const double mlo = n * fmax(0.0, double(wl) * 0.99 * double(a.fixscale) - 1.0);
          const double e = bin_err(1, eps, xmax_from(k0)) * mhi;
          ez += e;
          if (lbab < pZ) bl = b;      // mass strictly above b may still be short of p Z
          ub += mhi;
          if (bh < 0) {
            if (ub >= pZ) bh = b;
            else ea += e;              // bins above bh: summed in registers
          }
          lbab += mlo;
        }
        const bool ok = bh >= 0 && bl >= 0 && bl <= bh && bh - bl < kCand;
        s_cand = ok ? 1 : 0;
        s_bl = uint32_t(bl);
        s_bh = uint32_t(bh);
        s_EZ = ez;
        s_EA = ea;
        // floor bin for the fallback: the bins below it hold at most
        // count x (mass of the bin's highest key) < (1 - p) Z / 2 in total
        const double budget = 0.5 * (1.0 - double(a.top_p)) * double(Z);
        double below = 0.0;
        uint32_t fb = 0;
        for (uint32_t b = 0; b < 256; ++b) {
          const uint32_t khi = (b << (KB - 8)) | ((1u << (KB - 8)) - 1u);
          const float zhi = KO::value(khi);
          const float w = (zhi == zhi) ? ex2_approx(fminf(__fmaf_rn(zhi, a.c, -Kc), 1.0f)) : 0.0f;
          below += double(hcnt[b]) * (double(w) * 1.01 * double(a.fixscale) + 1.0);
          if (below >= budget) break;
          fb = b + 1;
        }
        s_floor = fb;
      }
      __syncthreads();
      if (s_cand) {
        // one pass: tokens above bh summed per thread, tokens in [bl, bh]
        // into a histogram of (top digit, second digit)
        const uint32_t bl = s_bl, bh = s_bh;
        unsigned long long* hsub = &hwarp[0][0];
        for (int i = tid; i < kCand * 256; i += NT) hsub[i] = 0;
        __syncthreads();
        unsigned long long ra = 0;
        sweep([&](float z) {
          const uint32_t k = KO::key(z), tb = k >> (KB - 8);
          if (tb > bh) {
            ra += mass(z);
          } else if (tb >= bl) {
            const unsigned long long q = mass(z);
            if (q) atomicAdd(&hsub[(tb - bl) * 256u + ((k >> (KB - 16)) & 255u)], q);
          }
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ra += __shfl_xor_sync(0xffffffffu, ra, o);
        if (lane == 0) s_red[warp] = ra;
        __syncthreads();
        if (tid == 0) {
          unsigned long long A = 0;
          for (int w = 0; w < NT / 32; ++w) A += s_red[w];
          const double target = double(a.top_p) * double(s_ztot);
          double EA = s_EA;
          uint32_t key16 = 0;
          unsigned long long mb = 0;
          bool found = false;
          for (int tb = int(bh); tb >= int(bl) && !found; --tb) {
            for (int d = 255; d >= 0; --d) {
              const unsigned long long m = hsub[(tb - int(bl)) * 256 + d];
              const uint32_t k16 = (uint32_t(tb) << 8) | uint32_t(d);
              if (double(A + m) >= target) {
                key16 = k16;
                mb = m;
                found = true;
                break;
              }
              A += m;
              EA += bin_err(m, eps, xmax_from(k16 << (KB - 16)));
            }
          }
          s_pre16 = key16;
          s_A = A;
          s_EA = EA;
          s_mb = mb;
          s_Z = s_ztot;
        }
        __syncthreads();
      } else {
        const uint32_t fb = s_floor;
        clear();
        for (int i = tid; i < (NT / 32) * 256; i += NT) (&hwarp[0][0])[i] = 0;
        __syncthreads();
        // a private histogram per warp: the few hot bins are not shared by
        // all warps' atomics
        sweep([&](float z) {
          const uint32_t k = KO::key(z);
          if ((k >> (KB - 8)) >= fb) {
            const unsigned long long q = mass(z);
            if (q) atomicAdd(&hwarp[warp][k >> (KB - 8)], q);
          }
        });
        __syncthreads();
        for (int b = tid; b < 256; b += NT) {
          unsigned long long m = 0;
          for (int w = 0; w < NT / 32; ++w) m += hwarp[w][b];
          hmass[b] = m;
        }
      }
    }
    __syncthreads();
    const bool cand = !topk && s_cand;
    if (tid == 0 && !cand) {
      unsigned long long Z = 0;
      double EZ = 0.0;
      for (int b = 0; b < 256; ++b) {
        Z += hmass[b];
        EZ += bin_err(hmass[b], eps, xmax_from(uint32_t(b) << (KB - 8)));
      }
      if (!topk) {  // the bins below the floor: in the total, not in the histogram
        EZ += bin_err(s_ztot - Z, eps, 200.0f);
        Z = s_ztot;
      }
      s_Z = Z;
      s_EZ = EZ;
      s_A = 0;
      s_EA = 0.0;
    }
    __syncthreads();
    const double target = double(a.top_p) * double(s_Z);
    uint32_t pre = cand ? s_pre16 : 0;
    for (int lvl = cand ? 2 : 0; lvl < ND; ++lvl) {
      const int sh = KB - 8 * (lvl + 1);
      if (lvl > 0) {
        const bool reuse = topk && lvl == ND - 1 && pre == (KA >> 8);
        __syncthreads();
        if (reuse) {
          for (int i = tid; i < 256; i += NT) hmass[i] = hbuck[i];
        } else {
          for (int i = tid; i < (NT / 32) * 256; i += NT) (&hwarp[0][0])[i] = 0;
          __syncthreads();
          sweep([&](float z) {
            const uint32_t k = KO::key(z);
            if (k >= KA && (k >> (sh + 8)) == pre) {
              const unsigned long long q = mass(z);
              if (q) atomicAdd(&hwarp[warp][(k >> sh) & 255u], q);
            }
          });
          __syncthreads();
          for (int b = tid; b < 256; b += NT) {
            unsigned long long m = 0;
            for (int w = 0; w < NT / 32; ++w) m += hwarp[w][b];
            hmass[b] = m;
          }
        }
        __syncthreads();
      }
      if (tid == 0) {
        unsigned long long A = s_A;
        double EA = s_EA;
        uint32_t d = 0;
        for (int b = 255; b >= 0; --b) {
          if (double(A + hmass[b]) >= target) {
            d = uint32_t(b);
            break;
          }
          A += hmass[b];
          EA += bin_err(hmass[b], eps, xmax_from(((pre << 8) | uint32_t(b)) << sh));
        }
        s_digit = d;
        s_A = A;
        s_EA = EA;
        s_mb = hmass[d];
      }
      __syncthreads();
      pre = (pre << 8) | s_digit;
    }
    if (tid == 0) {
      // certify: mass(keys >= K) >= p Z and mass(keys > K) < p Z hold exactly
      const double C = double(s_A + s_mb), Cm = double(s_A);
      const double q = 2.0 * double(a.V) + 2.0;  // rounding to fixed point
      const double EC = s_EA + bin_err(s_mb, eps, xmax_from(pre)) + q;
      const double ECm = s_EA + q;
      const double Zlo = double(s_Z) - s_EZ - q, Zhi = double(s_Z) + s_EZ + q;
      const bool ok = (C - EC >= double(a.top_p) * Zhi) && (Cm + ECm < double(a.top_p) * Zlo);
      const float tp = KO::value(pre);
      a.out[row] = (ok || kAcc) ? fmaxf(tau, tp) : NAN;
    }
    return;
  }
  if (tid == 0) a.out[row] = tau;
}

// ---------------------------------------------------------------- bf16 rows
// bf16 rows with top-k or top-p on, two passes per row. Pass A takes the row
// maximum (NaN propagates). Pass B counts the logits within 255 keys of the
// maximum's key, one shared-memory bin per key, so that a bin holds one logit
// value exactly and the logits outside the window cost one compare. Top-k:
// the k-th largest logit is the bin where the count from the top reaches k;
// top-p on the kept tokens needs only their masses, count x exp((v - max) /
// T) per bin, in fp64 with sums formed by additions from the top. Top-p
// alone: pass B also sums the fp32 masses below the window, and the bin where
// the window's mass from the top reaches p Z is taken when the comparison
// holds within the error bounds of both parts. A row the kernel cannot settle
// (fewer than k logits in the window, the top-p boundary below it, or an
// uncertified comparison) gets NaN and the general kernel takes it.
// Persistent CTAs, three per SM (measured faster than one, two, or more
// smaller ones), walk the rows; a row read by pass A is still in L2 for
// pass B.
constexpr int kFTK = 512;

// Relative error bound of one fp32 mass 2^x outside the window (pass B, top-p
// alone): ex2.approx, the two roundings of x = (z Chi - Kc) + z Clo (ln2 u |x|
// with |x| <= 127 for every term not flushed) and the truncation of C to
// Chi + Clo (below 1e-9 for offsets under 2^18); the vector tree (3u) and the
// compensated running sum (below 2u) on top.
constexpr double kOutRelErr = 1.6e-7 * 1.1 + 0.6931471805599453 * 5.9604644775390625e-8 * 128.0 +
                              1e-9 + 5.0 * 5.9604644775390625e-8;

template <bool kPAlone>
__global__ void __launch_bounds__(kFTK, 3) filter_topk_bf16_kernel(const FilterArgs a) {
  using KO = KeyOf<EBf16>;
  __shared__ uint32_t hist[256];
  __shared__ float s_m[kFTK / 32];
  __shared__ double s_zo[kFTK / 32];
  __shared__ float s_th[kPAlone ? 256 : 1], s_tl[kPAlone ? 256 : 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned full = 0xffffffffu;
  const bool topp = a.top_p < 1.0f;
  if (kPAlone) {
    for (int j = tid; j < 256; j += kFTK) {
      s_th[j] = kExp2Tab.hi[j];
      s_tl[j] = kExp2Tab.lo[j];
    }
  }
  for (int row = blockIdx.x; row < a.R; row += gridDim.x) {
    const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const char*>(a.logits) +
                                                     size_t(row) * size_t(a.V) * 2);
    // pass A: row maximum
    float vm = -INFINITY;
    int i = tid;
    for (; i + 3 * kFTK < a.nvec; i += 4 * kFTK) {  // four loads in flight per thread
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = ldg_nc_v4(rp + i + u * kFTK);
#pragma unroll
      for (int u = 0; u < 4; ++u) vm = max_nan(vm, EBf16::vmax(v[u]));
    }
    for (; i < a.nvec; i += kFTK) vm = max_nan(vm, EBf16::vmax(ldg_nc_v4(rp + i)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vm = max_nan(vm, __shfl_xor_sync(full, vm, o));
    if (lane == 0) s_m[warp] = vm;
    for (int j = tid; j < 256; j += kFTK) hist[j] = 0;
    __syncthreads();
    float mx = s_m[0];
    for (int w = 1; w < kFTK / 32; ++w) mx = max_nan(mx, s_m[w]);
    const float Kc = offset_of(mx, a.c);
    const bool nan_row = mx != mx;
    const bool range_bad = topp && mx > -INFINITY && !(fabsf(Kc) < kMaxOffset);
    if (nan_row || range_bad || !(mx > -INFINITY)) {
      if (tid == 0) {
        a.out[row] = (nan_row || range_bad) ? INFINITY : -INFINITY;
        if ((nan_row || range_bad) && a.err) atomicOr(a.err, SPEC_DERR_LOGITS);
      }
      __syncthreads();  // s_m is written again for the next row
      continue;
    }
    // the maximum's key (+0 when the maximum is a zero: -0 and +0 are both in)
    const uint32_t mk = (mx == 0.0f) ? 0x8000u : KO::key(mx);
    const uint32_t lo = mk >= 255u ? mk - 255u : 0u;
    // pass B: exact counts of the keys in [lo, mk]; with top-p alone also the
    // mass of the logits below the window, 2^(z C - Kc) in fp32 (compensated)
    float zo = 0.0f, zol = 0.0f;
    auto count = [&](const uint4& v) {
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      float m[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const uint32_t b = (w4[h >> 1] >> (16 * (h & 1))) & 0xffffu;
        const uint32_t k = (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
        if (k >= lo) atomicAdd(&hist[k - lo], 1u);
        if (kPAlone) {
          const float z = __uint_as_float(b << 16);
          const float x = __fmaf_rn(z, a.Clo, __fmaf_rn(z, a.Chi, -Kc));
          m[h] = (k >= lo) ? 0.0f : ex2_approx(x);
        }
      }
      if (kPAlone) {
#pragma unroll
        for (int w = 1; w < 8; w <<= 1)
#pragma unroll
          for (int h = 0; h < 8; h += 2 * w) m[h] = __fadd_rn(m[h], m[h + w]);
        const df t = two_sum(zo, m[0]);
        zo = t.hi;
        zol = __fadd_rn(zol, t.lo);
      }
    };
    i = tid;
    for (; i + 3 * kFTK < a.nvec; i += 4 * kFTK) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = ldg_nc_v4(rp + i + u * kFTK);
#pragma unroll
      for (int u = 0; u < 4; ++u) count(v[u]);
    }
    for (; i < a.nvec; i += kFTK) count(ldg_nc_v4(rp + i));
    if (kPAlone) {
      double d = double(zo) + double(zol);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(full, d, o);
      if (lane == 0) s_zo[warp] = d;
    }
    __syncthreads();
    if (warp == 0) {
      float out = NAN;  // the general kernel takes the rows left NaN
      if (!kPAlone) {
        // top-k (then top-p on the kept tokens): lane l holds bins 8l .. 8l + 7
        uint32_t c[8], s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[lane * 8 + j];
          s += c[j];
        }
        uint32_t S = s;  // count in the bins of lanes >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_down_sync(full, S, o);
          if (lane + o < 32) S += t;
        }
        const uint32_t need = uint32_t(a.top_k);
        const unsigned bal = __ballot_sync(full, S >= need);
        if (bal != 0) {  // else fewer than k logits in the window
          const int L = 31 - __clz(int(bal));
          int tb = -1;  // highest bin whose count from the top reaches k
          if (lane == L) {
            uint32_t suf = S;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (suf >= need) tb = 8 * L + j;
              suf -= c[j];
            }
          }
          tb = __shfl_sync(full, tb, L);
          int pb = tb;
          if (topp) {
            // kept bins tb .. 255, bin 255 - lane - 32 m in lane `lane`: masses
            // count x exp((v - max) / T) in fp64, one exponential per lane for
            // up to 32 kept bins
            double e[8], zs = 0.0;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int b = 255 - lane - 32 * m;
              e[m] = 0.0;
              if (b >= tb) {
                const uint32_t cb = hist[b];
                if (cb != 0u)
                  e[m] = double(cb) *
                         exp((double(KO::value(lo + uint32_t(b))) - double(mx)) / double(a.T));
              }
              zs += e[m];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(full, zs, o);
            const double target = double(a.top_p) * zs;
            // mass from the top, bin by bin: the highest bin where it reaches p Z
            double carry = 0.0;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              if (255 - 32 * m < tb) break;
              double inc = e[m];
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const double t = __shfl_up_sync(full, inc, o);
                if (lane >= o) inc += t;
              }
              const int b = 255 - lane - 32 * m;
              const unsigned hit = __ballot_sync(full, b >= tb && carry + inc >= target);
              if (hit) {
                pb = 255 - (__ffs(int(hit)) - 1) - 32 * m;
                break;
              }
              carry += __shfl_sync(full, inc, 31);
            }
          }
          out = KO::value(lo + uint32_t(pb));
        }
      } else {
        // top-p alone: window masses count x 2^(v C - Kc) in pair arithmetic
        // (relative error below acc_rho), the mass below the window from pass
        // B (relative error below kOutRelErr); the bin is taken when the
        // comparisons with p Z hold for every value within those bounds
        double e[8], zs = 0.0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int b = 255 - lane - 32 * m;
          const uint32_t cb = hist[b];
          e[m] = 0.0;
          if (cb != 0u) {
            const float v = KO::value(lo + uint32_t(b));
            const df p = two_prod(v, a.Chi);
            const float pl = __fmaf_rn(v, a.Clo, p.lo);
            const df sx = two_sum(p.hi, -Kc);
            const df r = df_exp2(sx.hi, __fadd_rn(sx.lo, pl), s_th, s_tl);
            e[m] = double(cb) * (double(r.hi) + double(r.lo));
          }
          zs += e[m];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(full, zs, o);
        double zo = lane < kFTK / 32 ? s_zo[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zo += __shfl_xor_sync(full, zo, o);
        const double Z = zs + zo;
        const double ew = 2e-12 + 2.2e-14 * (fabs(double(Kc)) + 256.0);
        const double err = zs * ew + zo * kOutRelErr * 1.05 + Z * 1e-15;
        const double target = double(a.top_p) * Z;
        double carry = 0.0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          double inc = e[m];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const double t = __shfl_up_sync(full, inc, o);
            if (lane >= o) inc += t;
          }
          const unsigned hit = __ballot_sync(full, carry + inc >= target);
          if (hit) {
            const int f = __ffs(int(hit)) - 1;
            const double incl = carry + __shfl_sync(full, inc, f);
            const double excl = incl - __shfl_sync(full, e[m], f);
            const double slack = zs * ew + 1e-15 * Z;
            const bool ok = incl - slack >= double(a.top_p) * (Z + err) &&
                            excl + slack < double(a.top_p) * (Z - err);
            if (ok) out = KO::value(lo + uint32_t(255 - f - 32 * m));
            break;
          }
          carry += __shfl_sync(full, inc, 31);
        }
      }
      if (lane == 0) a.out[row] = out;
    }
    __syncthreads();
  }
}

}  // namespace

int launch_filter(const FilterLaunch& f) {
  FilterArgs a;
  a.logits = f.logits;
  a.R = f.R;
  a.V = f.V;
  const int kvec = (f.dtype == SPEC_BF16) ? 8 : 4;
  a.nvec = f.V / kvec;
  a.top_k = f.top_k;
  a.top_p = f.top_p;
  a.T = f.temperature;
  a.skip_done = 0;
  const double C = 1.4426950408889634073599246810018921 / double(f.temperature);
  a.c = float(C);
  a.Chi = float(C);
  a.Clo = float(C - double(a.Chi));
  a.ex2 = float(kEx2RelErrBound);
  // fixed-point scale 2^s with 2 V 2^s < 2^63 (each mass is at most 2)
  int lg = 0;
  while ((1 << lg) < f.V) ++lg;
  a.fixscale = std::ldexp(1.0f, 61 - lg);
  a.out = f.out;
  a.err = f.err;
  cudaStream_t st = static_cast<cudaStream_t>(f.stream);
  if (f.dtype == SPEC_BF16) {
    const bool topk = f.top_k > 0 && f.top_k < f.V;
    if (topk || f.top_p < 1.0f) {
      int dev = 0, sms = 0;  // a cheap attribute query on every call: no shared host state
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (sms < 1) sms = 1;
      const int grid = f.R < 3 * sms ? f.R : 3 * sms;
      if (topk) filter_topk_bf16_kernel<false><<<grid, kFTK, 0, st>>>(a);
      else filter_topk_bf16_kernel<true><<<grid, kFTK, 0, st>>>(a);
      a.skip_done = 1;
    }
    filter_kernel<EBf16, false><<<f.R, kFT, 0, st>>>(a);
    if (f.top_p < 1.0f) filter_kernel<EBf16, true><<<f.R, kFTAcc, 0, st>>>(a);
  } else {
    filter_kernel<EF32, false><<<f.R, kFT, 0, st>>>(a);
    if (f.top_p < 1.0f) filter_kernel<EF32, true><<<f.R, kFTAcc, 0, st>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // namespace sv
