// Double-float ("float-float") arithmetic and an accurate base-2 exponential
// built only on fp32 FMA-pipe instructions.
//
// GB300 runs fp64 at a small fraction of its fp32 rate, so the high-precision
// path of the sampler works on unevaluated sums hi + lo of two floats
// (Dekker / Knuth error-free transformations). The exponential follows the
// table-driven method of P. T. P. Tang ("Table-driven implementation of the
// exponential function in IEEE floating-point arithmetic", ACM TOMS 15(2),
// 1989): 2^x = 2^m * 2^(j/256) * exp(t), |t| <= ln2/512, with the 256 table
// values held as hi + lo pairs and exp(t) - 1 from its Taylor series.
//
// Error: every result here carries a relative error below kDfExpRelErr
// (derivation next to df_exp2), far below fp32's 6e-8.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace sv {

struct df {
  float hi, lo;
};

// s + e == a + b exactly (Knuth's TwoSum, no ordering requirement).
__device__ __forceinline__ df two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// s + e == a + b exactly when |a| >= |b| (Dekker's FastTwoSum).
__device__ __forceinline__ df fast_two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float e = __fsub_rn(b, __fsub_rn(s, a));
  return {s, e};
}

// p + e == a * b exactly (FMA-based TwoProduct).
__device__ __forceinline__ df two_prod(float a, float b) {
  float p = __fmul_rn(a, b);
  float e = __fmaf_rn(a, b, -p);
  return {p, e};
}

__device__ __forceinline__ df df_add(df x, df y) {
  df s = two_sum(x.hi, y.hi);
  float e = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
  return fast_two_sum(s.hi, e);
}

__device__ __forceinline__ df df_sub(df x, df y) { return df_add(x, df{-y.hi, -y.lo}); }

__device__ __forceinline__ df df_mul(df x, df y) {
  df p = two_prod(x.hi, y.hi);
  float e = __fmaf_rn(x.hi, y.lo, __fmaf_rn(x.lo, y.hi, p.lo));
  return fast_two_sum(p.hi, e);
}

__device__ __forceinline__ df df_add_f(df x, float y) {
  df s = two_sum(x.hi, y);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}

__device__ __forceinline__ df df_mul_f(df x, float y) {
  df p = two_prod(x.hi, y);
  return fast_two_sum(p.hi, __fmaf_rn(x.lo, y, p.lo));
}

// 1/x for x > 0: float reciprocal refined by one Newton step in pair arithmetic.
__device__ __forceinline__ df df_recip(df x) {
  const float r0 = __frcp_rn(x.hi);
  // e = 1 - x*r0 formed from the exact residual of x.hi*r0
  const float e = __fsub_rn(-__fmaf_rn(x.hi, r0, -1.0f), __fmul_rn(x.lo, r0));
  return fast_two_sum(r0, __fmul_rn(r0, e));
}

__device__ __forceinline__ bool df_gt(df a, df b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ df df_shfl_xor(df x, int o) {
  return {__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)};
}
__device__ __forceinline__ df df_shfl_up(df x, int o) {
  return {__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
}
__device__ __forceinline__ df df_shfl(df x, int l) {
  return {__shfl_sync(0xffffffffu, x.hi, l), __shfl_sync(0xffffffffu, x.lo, l)};
}

// Warp sum in pair arithmetic; df_add is commutative bit for bit (the error of
// TwoSum is exact), so every lane ends with the same value.
__device__ __forceinline__ df df_warp_sum(df v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
  return v;
}

// ---------------------------------------------------------------- 2^(j/256)
// Values computed at compile time in double precision from the exponential
// series (exp(y) = sum y^n/n!, y = j ln2 / 256 <= ln2, 30 terms: truncation
// below 1e-30), then split into float hi + lo (|lo| <= ulp(hi)/2).
struct Exp2Table {
  float hi[256];
  float lo[256];
};

constexpr double kLn2d = 0.693147180559945309417232121458176568;

constexpr double exp_series(double y) {
  double term = 1.0, sum = 1.0;
  for (int n = 1; n < 30; ++n) {
    term = term * y / n;
    sum += term;
  }
  return sum;
}

constexpr Exp2Table make_exp2_table() {
  Exp2Table t{};
  for (int j = 0; j < 256; ++j) {
    double v = exp_series(kLn2d * j / 256.0);
    float h = static_cast<float>(v);
    t.hi[j] = h;
    t.lo[j] = static_cast<float>(v - static_cast<double>(h));
  }
  return t;
}

__constant__ Exp2Table kExp2Tab = make_exp2_table();

// ln 2 as a float pair.
constexpr float kLn2Hi = 0.693147182464599609375f;               // fl32(ln 2)
constexpr float kLn2Lo = static_cast<float>(kLn2d - 0.693147182464599609375);

// 2^(xh + xl) as hi + lo, for xh + xl in [-126, 127). Smaller values return 0
// (an absolute error below 2^-126 per term, far below every error budget here).
//   m + j/256 = round(256 xh) / 256, g = xh - (m + j/256) is exact because
//   xh is a multiple of ulp(xh) <= 2^-16 (|xh| < 2^8), so is g, and |g| <= 2^-9;
//   t = (g + xl) ln2 is formed as a float pair (error < 2^-46 |t|);
//   exp(t) = 1 + t + t^2/2 + t^3/6 + t^4/24 with |t| < 1.37e-3 when |xl| <=
//   2^-16 (a normalised pair, or a term below 2^7 in magnitude): truncation
//   < 4e-17, the t^2.. part (< 9.4e-7) evaluated in fp32 (error < 2.3e-13);
//   the product with the table pair adds < 2^-46.
// Total relative error < kDfExpRelErr = 4e-13 when |xl| <= 2^-16. A larger xl
// (|t| <= ln2 (2^-9 + |xl|)) adds the truncation |t|^5/120 and an fp32 error
// below 1.5 u t^2: the caller's budget takes them (see acc_rho).
constexpr double kDfExpRelErr = 4e-13;

template <class Tab>
__device__ __forceinline__ df df_exp2_t(float xh, float xl, const Tab& tab);

// The table as two arrays (hi values, lo values).
struct SplitTab {
  const float* hi;
  const float* lo;
  __device__ __forceinline__ float2 operator[](int j) const { return make_float2(hi[j], lo[j]); }
};
// The table interleaved: element j = (hi, lo) of 2^(j/256), one 8-byte load.
struct PairTab {
  const float2* t;
  __device__ __forceinline__ float2 operator[](int j) const { return t[j]; }
};

__device__ __forceinline__ df df_exp2(float xh, float xl, const float* tab_hi,
                                      const float* tab_lo) {
  return df_exp2_t(xh, xl, SplitTab{tab_hi, tab_lo});
}
__device__ __forceinline__ df df_exp2(float xh, float xl, const float2* tab) {
  return df_exp2_t(xh, xl, PairTab{tab});
}

template <class Tab>
__device__ __forceinline__ df df_exp2_t(float xh, float xl, const Tab& tab) {
  if (!(xh >= -126.0f)) return {0.0f, 0.0f};  // below 2^-126 (or -inf): flushed
  float k = rintf(__fmul_rn(xh, 256.0f));
  float g = __fmaf_rn(k, -1.0f / 256.0f, xh);  // exact
  int ki = static_cast<int>(k);
  int j = ki & 255;
  int m = (ki - j) / 256;  // floor division (ki - j is a multiple of 256)
  // t = (g + xl) * ln2 as a pair
  df gl = two_sum(g, xl);
  float th = __fmul_rn(gl.hi, kLn2Hi);
  float tl = __fmaf_rn(gl.hi, kLn2Hi, -th);
  tl = __fmaf_rn(gl.hi, kLn2Lo, tl);
  tl = __fmaf_rn(gl.lo, kLn2Hi, tl);
  // exp(t) - 1 - t = t^2/2 + t^3/6 + t^4/24 (+ the cross term th*tl)
  float q = __fmaf_rn(th, 1.0f / 24.0f, 1.0f / 6.0f);
  q = __fmaf_rn(th, q, 0.5f);
  q = __fmul_rn(__fmul_rn(th, th), q);
  q = __fmaf_rn(th, tl, q);
  // e = 1 + th + (tl + q)
  df e = fast_two_sum(1.0f, th);
  e.lo = __fadd_rn(e.lo, __fadd_rn(tl, q));
  // r = T[j] * e
  const float2 T = tab[j];
  const float Th = T.x, Tl = T.y;
  float rh = __fmul_rn(Th, e.hi);
  float rl = __fmaf_rn(Th, e.hi, -rh);
  rl = __fmaf_rn(Th, e.lo, rl);
  rl = __fmaf_rn(Tl, e.hi, rl);
  df r = fast_two_sum(rh, rl);
  // scale by 2^m (exact: m >= -127 and the result stays normal or is flushed)
  if (m < -126) return {0.0f, 0.0f};
  float s = __int_as_float((m + 127) << 23);
  return {__fmul_rn(r.hi, s), __fmul_rn(r.lo, s)};
}

// ---------------------------------------------------------------- lighter exponential
// 2^(z C - Kc) for two logits at once, each with its own integer offset Kc,
// as an unevaluated pair e = hi + lo, with a relative error below
// kLiteExpRelErr: about a third of the instructions of df_exp2 (packed f32x2
// arithmetic, no pair arithmetic in the reduction or the polynomial) for a
// bound of 1e-9 instead of 4e-13. Valid while |z C| stays below 1100 for every
// term that is not flushed (callers take it only for rows whose offsets
// satisfy |Kc| <= kLiteMaxOffset; terms below 2^(Kc - 127) relative to the
// offset are flushed to 0, the clamp of z at zlo maps -inf and anything far
// below the offset there).
//
// Method (Tang's table reduction with 256 entries, as df_exp2):
//   ph + pl = z Chi exactly (FMA TwoProduct), t1 = fl(z Clo + pl);
//   n = rint(256 ph) from the magic-number addition (|256 ph| < 2^22), so
//   g = ph - n/256 is exact and |g| <= 2^-9;
//   r = fl(g + t1): error below u |r| <= 2^-33 (|t1| <= 2u |ph| < 1.4e-4);
//   2^r - 1 = p(r) = r (c1 + r (c2 + r c3)), Taylor to the cubic term
//   (truncation < 2e-13 for |r ln2| < 1.5e-3), three roundings and the
//   float coefficients: absolute error < 2.7e-10;
//   2^(j/256) from the pair table (2^-48), lo = fl(T.hi p + T.lo): rounding
//   < 1.8e-10 relative, the dropped T.lo p < 9e-11;
//   the scaling by 2^(m - Kc), m = floor(n / 256), is exact.
// Sum of the parts, with z C's own representation error (2^-48 |z C|) and
// the rounding of t1: below 7e-10 for |z C| < 1100; kLiteExpRelErr = 1e-9.
constexpr double kLiteExpRelErr = 1e-9;
constexpr float kLiteMaxOffset = 896.0f;  // |Kc| <= 896: |z C| <= 1056 for every term kept

struct LiteConsts {
  uint64_t chi2, nchi2, clo2;  // (Chi, Chi), (-Chi, -Chi), (Clo, Clo)
};

__device__ __forceinline__ LiteConsts lite_consts(float Chi, float Clo) {
  return {f2_pack(Chi, Chi), f2_pack(-Chi, -Chi), f2_pack(Clo, Clo)};
}

// Per-lane row constants: the lowest logit kept for offset Kc (terms of
// smaller z are below 2^-150 of the offset and flush; clamping there also maps
// -inf to a flushed term) and the exponent bias 127 - Kc.
struct LiteRow {
  float zlo;
  int bias;
};
__device__ __forceinline__ LiteRow lite_row(float Kc, float Chi) {
  return {__fdiv_rn(__fsub_rn(Kc, 160.0f), Chi), 127 - static_cast<int>(Kc)};
}

// e0 = 2^(z0 C - K0), e1 = 2^(z1 C - K1) with the rows' constants R0, R1;
// tab the interleaved 2^(j/256) table.
__device__ __forceinline__ void lite_exp2x2(float z0, float z1, const LiteRow& R0,
                                            const LiteRow& R1, const LiteConsts& C,
                                            const float2* tab, df& e0, df& e1) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const uint64_t magic2 = f2_pack(kMagic, kMagic);
  const uint64_t z2 = f2_pack(fmaxf(z0, R0.zlo), fmaxf(z1, R1.zlo));
  const uint64_t nph = f2_mul(z2, C.nchi2);                         // -ph
  const uint64_t pl = f2_fma(z2, C.chi2, nph);                      // z Chi - ph, exact
  const uint64_t t1 = f2_fma(z2, C.clo2, pl);                       // z Clo + pl
  const uint64_t nb = f2_fma(nph, f2_pack(-256.0f, -256.0f), magic2);  // magic + rint(256 ph)
  const uint64_t nf = f2_sub(nb, magic2);                           // rint(256 ph)
  const uint64_t gneg = f2_fma(nf, f2_pack(1.0f / 256.0f, 1.0f / 256.0f), nph);  // -g, exact
  const uint64_t r = f2_sub(t1, gneg);                              // g + t1
  const uint64_t in = f2_fma(r, f2_pack(0.0555041086648215799531422637686f,
                                        0.0555041086648215799531422637686f),
                             f2_pack(0.240226506959100712333551263163f,
                                     0.240226506959100712333551263163f));
  const uint64_t mid = f2_fma(r, in, f2_pack(0.693147180559945309417232121458f,
                                             0.693147180559945309417232121458f));
  const uint64_t pr = f2_mul(r, mid);                               // 2^r - 1
  float nb0, nb1;
  f2_unpack(nb, nb0, nb1);
  const int n0 = __float_as_int(nb0) - __float_as_int(kMagic);
  const int n1 = __float_as_int(nb1) - __float_as_int(kMagic);
  const float2 T0 = tab[n0 & 255], T1 = tab[n1 & 255];
  const uint64_t th = f2_pack(T0.x, T1.x);
  const uint64_t lo = f2_fma(th, pr, f2_pack(T0.y, T1.y));
  // 2^(m - K), m = n >> 8 (arithmetic, i.e. floor(n / 256)): exponent field
  // m - K + 127; a field <= 0 flushes the term
  const int b0 = max((n0 >> 8) + R0.bias, 0) << 23;
  const int b1 = max((n1 >> 8) + R1.bias, 0) << 23;
  const uint64_t sc = f2_pack(__int_as_float(b0), __int_as_float(b1));
  float h0, h1, l0, l1;
  f2_unpack(f2_mul(th, sc), h0, h1);
  f2_unpack(f2_mul(lo, sc), l0, l1);
  e0 = {h0, l0};
  e1 = {h1, l1};
}

}  // namespace sv
