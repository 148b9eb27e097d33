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

__device__ __forceinline__ df df_exp2(float xh, float xl, const float* tab_hi,
                                      const float* tab_lo) {
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
  float Th = tab_hi[j], Tl = tab_lo[j];
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

}  // namespace sv
