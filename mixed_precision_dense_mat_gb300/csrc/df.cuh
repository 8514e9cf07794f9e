// Double-float arithmetic: a value is the unevaluated sum hi + lo of two FP32 numbers
// (about 48 significant bits).  Built from the error-free transformations of Dekker
// ("A floating-point technique for extending the available precision", Numer. Math. 18,
// 1971) and Knuth (two-sum, TAOCP vol. 2): two_sum returns a + b exactly as s + e,
// two_prod returns a * b exactly as p + e using one fused multiply-add.  Intrinsics with
// explicit rounding keep the compiler from contracting or reordering these steps.
// Used where GB300's FP64 units (about 1/60 of the FP32 rate) would otherwise bound a
// kernel and ~1e-14 relative accuracy is enough.
#pragma once

namespace cr {

struct df {
  float hi, lo;
};

__device__ __forceinline__ df df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
// requires |a| >= |b| (or a == 0)
__device__ __forceinline__ df df_quick_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ df df_two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ df df_add(df x, df y) {
  const df s = df_two_sum(x.hi, y.hi);
  const float e = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
  return df_quick_two_sum(s.hi, e);
}
__device__ __forceinline__ df df_add_f(df x, float y) {
  const df s = df_two_sum(x.hi, y);
  return df_quick_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}
__device__ __forceinline__ df df_neg(df x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ df df_mul(df x, df y) {
  const df p = df_two_prod(x.hi, y.hi);
  const float e = __fmaf_rn(x.hi, y.lo, __fmaf_rn(x.lo, y.hi, p.lo));
  return df_quick_two_sum(p.hi, e);
}
__device__ __forceinline__ df df_mul_f(df x, float y) {
  const df p = df_two_prod(x.hi, y);
  return df_quick_two_sum(p.hi, __fmaf_rn(x.lo, y, p.lo));
}
// x * 2^e for -126 <= e <= 127 (exact unless the low part becomes subnormal)
__device__ __forceinline__ df df_ldexp(df x, int e) {
  const float s = __int_as_float((e + 127) << 23);
  return {__fmul_rn(x.hi, s), __fmul_rn(x.lo, s)};
}
__host__ __device__ __forceinline__ df df_from_double(double d) {
  const float h = (float)d;
  return {h, (float)(d - (double)h)};
}
__device__ __forceinline__ double df_to_double(df x) { return (double)x.hi + (double)x.lo; }
__device__ __forceinline__ bool df_lt(df a, df b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }

// sqrt of a non-negative double-float: FP32 square root refined by one Newton step whose
// residual d - s^2 is formed exactly.  The step's coefficient 1/(2s) scales a correction of
// relative size ~2^-24, so the approximate reciprocal (relative error ~2^-22) is ample.
__device__ __forceinline__ df df_sqrt(df d) {
  if (d.hi <= 0.0f) return {0.0f, 0.0f};
  const float s = __fsqrt_rn(d.hi);
  const df p = df_two_prod(s, s);
  const float r = __fadd_rn(__fsub_rn(__fsub_rn(d.hi, p.hi), p.lo), d.lo);
  float inv_s;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv_s) : "f"(s));
  return df_quick_two_sum(s, __fmul_rn(r, 0.5f * inv_s));
}

// Constants of df_exp: 2^(j/64) as double-float pairs and ln2/64 in three pieces, the first
// with 11 significant bits so that k * piece is exact for |k| < 2^13.
struct DfExpTables {
  float t_hi[64], t_lo[64];
  float c1, c2, c3;
};

// exp(y) for -80 <= y <= 0 (callers route larger distances elsewhere), by Tang's
// table-driven method (P. T. P. Tang, "Table-driven implementation of the exponential function
// in IEEE floating-point arithmetic", ACM TOMS 15(2), 1989) carried out in double-float:
// y = k ln2/64 + r with |r| <= ln2/128, k = 64 m + j; exp(y) = 2^m 2^(j/64) exp(r), and
// exp(r) = 1 + r + r^2/2 + (r^3/6 + r^4/24 + r^5/120) with the bracket in FP32 (its
// magnitude is below 3e-8, so its FP32 rounding stays near 1e-15 of the result).
__device__ __forceinline__ df df_exp(df y, const DfExpTables& T) {
  // k = round(y 64 / ln 2) by adding 1.5 2^23 (exact rounding to nearest for |v| < 2^22):
  // FADD and integer work only, no conversion instruction
  const float big = 12582912.0f;
  const float kb = __fadd_rn(__fmul_rn(y.hi, 92.33248261689366f), big);   // 64 / ln 2
  const float kf = __fsub_rn(kb, big);
  const int k = __float_as_int(kb) - __float_as_int(big);
  const float t = __fmaf_rn(-kf, T.c1, y.hi);                     // exact (see above)
  df r = df_two_sum(t, y.lo);
  r = df_add(r, df_neg(df_two_prod(kf, T.c2)));
  r = df_add_f(r, -__fmul_rn(kf, T.c3));
  const float x = r.hi;
  const float q = __fmul_rn(__fmul_rn(x, __fmul_rn(x, x)),
                            __fmaf_rn(x, __fmaf_rn(x, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f));
  const df x2 = df_two_prod(x, x);
  const df half_r2 = {0.5f * x2.hi, 0.5f * __fmaf_rn(2.0f * x, r.lo, x2.lo)};
  df s = df_add(r, half_r2);
  s = df_add_f(s, q);
  df e = df_quick_two_sum(1.0f, s.hi);
  e = df_quick_two_sum(e.hi, __fadd_rn(e.lo, s.lo));
  const int j = k & 63;
  const int m = (k - j) / 64;
  const df tj = {T.t_hi[j], T.t_lo[j]};
  return df_ldexp(df_mul(tj, e), m);
}

// exp(y) for -80 <= y <= 0 to about 2^-39 relative, for values that are rounded to FP32
// afterwards: the reduction of df_exp with the last piece of ln2/64 folded into the low
// part, and exp(r) = 1 + r_hi + (r_lo + r_hi^2/2 + r_hi^3/6 + r_hi^4/24) with the bracket in
// FP32 (|r| <= ln2/128, so the bracket is below 1.5e-5 and its FP32 rounding below 2^-39; the
// omitted r^5/120 is below 2^-44).
__device__ __forceinline__ df df_exp_lite(df y, const DfExpTables& T) {
  const float big = 12582912.0f;
  const float kb = __fadd_rn(__fmul_rn(y.hi, 92.33248261689366f), big);   // 64 / ln 2
  const float kf = __fsub_rn(kb, big);
  const int k = __float_as_int(kb) - __float_as_int(big);
  const float t = __fmaf_rn(-kf, T.c1, y.hi);                     // exact
  const df p = df_two_prod(kf, T.c2);
  const df s = df_two_sum(t, -p.hi);
  const float lo = __fmaf_rn(-kf, T.c3, __fsub_rn(__fadd_rn(s.lo, y.lo), p.lo));
  const df r = df_two_sum(s.hi, lo);   // |lo| may exceed a tiny reduced argument
  const float x = r.hi;
  const float q = __fmul_rn(__fmul_rn(x, x), __fmaf_rn(x, __fmaf_rn(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f));
  df e = df_quick_two_sum(1.0f, x);
  e = df_quick_two_sum(e.hi, __fadd_rn(e.lo, __fadd_rn(r.lo, q)));
  const int j = k & 63;
  const int m = (k - j) / 64;
  const df tj = {T.t_hi[j], T.t_lo[j]};
  return df_ldexp(df_mul(tj, e), m);
}

}  // namespace cr
