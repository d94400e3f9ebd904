// Evaluation of one entry of the per-head distance tables (see table.cu),
// shared by the table kernel and the backward preprocess.
#pragma once

#include "bam_common.cuh"

namespace bam {

// b, db/dbeta and db/dmu at distance d, in fp32 arithmetic only (fp64 is slow
// on this GPU).  The exponent y = beta * log2(u / alpha) is carried as an
// unevaluated sum of two floats: log2(u/alpha) = e + log2(m) with the exact
// binary exponent e and the mantissa m in [0.5, 1) (log2f(m) has an absolute
// error ~6e-8), the products beta*e and beta*log2(m) are split exactly with
// fma, and the sum with TwoSum.  2^y is then 2^n (exact) times exp2f of the
// small remainder, so the relative error of b stays a few 1e-7 at any
// magnitude, where a plain fp32 pow loses ~1e-7 * |y| (1e-6 at |b| ~ 1e4).
// The theta prior of the BAM README ("Implementation Details"):
//   b = -exp(ta) * w^tb,  w = |d - mu| + eps,  mu = exp(tm) - exp(-tm),
// evaluated as -2^y with y = tb * log2(w) + ta * log2(e), by the same
// compensated exponent (ta * log2(e) split with a two-float log2(e)).  Also
// db/dtb = b ln(w) and db/dtm = -tb b sgn(d - mu) / w * (exp(tm) + exp(-tm)).
// eps > 0, so w > 0.
template <bool kGrads>
__device__ __forceinline__ void bias_terms_theta(int dint, float ta, float tb, float tm,
                                                 float eps, float* b, float* dtb, float* dtm) {
  const float muv = 2.0f * sinhf(tm);
  const float dm = static_cast<float>(dint) - muv;
  const float w = fabsf(dm) + eps;
  int e2 = 0;
  const float mant = frexpf(w, &e2);  // w = mant * 2^e2
  const float lm = log2f(mant);
  const float fe = static_cast<float>(e2);
  constexpr float kL2eHi = 1.44269502162933349609375f;  // fp32 log2(e)
  constexpr float kL2eLo = 1.925962989091e-08f;          // log2(e) - kL2eHi
  const float p1 = tb * fe, q1 = fmaf(tb, fe, -p1);
  const float p2 = tb * lm, q2 = fmaf(tb, lm, -p2);
  const float p3 = ta * kL2eHi, q3 = fmaf(ta, kL2eHi, -p3) + ta * kL2eLo;
  // TwoSum(p1, p2), then TwoSum(that, p3)
  const float s1 = p1 + p2;
  const float v1 = s1 - p1;
  const float e1 = (p1 - (s1 - v1)) + (p2 - v1);
  const float s2 = s1 + p3;
  const float v2 = s2 - s1;
  const float e2s = (s1 - (s2 - v2)) + (p3 - v2);
  float yh = s2, yl = e1 + e2s + q1 + q2 + q3;
  yh = fminf(fmaxf(yh, -400.0f), 400.0f);
  const float n = floorf(yh);
  const float f = (yh - n) + yl;
  const float bb = -ldexpf(exp2f(f), static_cast<int>(n));
  *b = bb;
  if (!kGrads) return;
  // ln w: near w = 1 the sum fe + lm cancels, so there ln w = log1p(w - 1)
  // with w - 1 = (|d - mu| - 1) + eps, whose first difference is exact.
  const float t = fabsf(dm);
  const float lnw = (t > 0.5f && t < 1.5f) ? log1pf((t - 1.0f) + eps)
                                          : (fe + lm) * 0.69314718055994530942f;
  *dtb = bb * lnw;  // b ln w
  const float sgn = dm > 0.0f ? 1.0f : (dm < 0.0f ? -1.0f : 0.0f);
  *dtm = -tb * bb * sgn / w * (2.0f * coshf(tm));
}

// kGrads: also the two derivatives (backward tables only).
template <bool kGrads>
__device__ __forceinline__ void bias_terms(int dint, float alpha, float beta, float mu, float eps,
                                           int prior, float* b, float* dbeta, float* dmu) {
  if (prior == kPriorTheta) {
    bias_terms_theta<kGrads>(dint, alpha, beta, mu, eps, b, dbeta, dmu);
    return;
  }
  float u = fabsf(static_cast<float>(dint) - mu);
  bool clamped = false;
  if (beta <= 0.0f && u < eps) {
    u = eps;
    clamped = true;
  }
  if (u == 0.0f) {
    *b = 0.0f;
    *dbeta = 0.0f;
    *dmu = 0.0f;
    return;
  }
  const float r = __fdiv_rn(u, alpha);
  int e2 = 0;
  const float mant = frexpf(r, &e2);  // r = mant * 2^e2
  const float lm = log2f(mant);
  const float fe = static_cast<float>(e2);
  // beta * fe and beta * lm with their rounding errors
  const float p1 = beta * fe, q1 = fmaf(beta, fe, -p1);
  const float p2 = beta * lm, q2 = fmaf(beta, lm, -p2);
  // TwoSum of p1 + p2
  const float sh = p1 + p2;
  const float bv = sh - p1;
  const float sl = (p1 - (sh - bv)) + (p2 - bv);
  float yh = sh, yl = sl + q1 + q2;  // y = yh + yl
  yh = fminf(fmaxf(yh, -400.0f), 400.0f);
  const float n = floorf(yh);
  const float f = (yh - n) + yl;  // yh - n is exact
  const float pw = ldexpf(exp2f(f), static_cast<int>(n));  // 2^y
  const float bb = -pw;
  *b = bb;
  if (!kGrads) return;
  // ln r: near r = 1 the sum fe + lm cancels, so there ln r = log1p((u - alpha)
  // / alpha), whose difference is exact.
  const float lnr = (u > 0.5f * alpha && u < 1.5f * alpha)
                        ? log1pf(__fdiv_rn(u - alpha, alpha))
                        : (fe + lm) * 0.69314718055994530942f;
  *dbeta = bb * lnr;  // b ln r
  const float sgn = (static_cast<float>(dint) - mu > 0.0f) ? 1.0f : -1.0f;
  *dmu = clamped ? 0.0f : -beta * bb * sgn / u;
}

__device__ __forceinline__ float to_f32_finite(float f) {
  // Keep the table finite so that exp2 of a difference never sees inf - inf.
  if (f < -3.0e38f) f = -3.0e38f;
  if (f > 3.0e38f) f = 3.0e38f;
  return f;
}

// Entry x of head h (see TableArgs).  Shared with the backward preprocess,
// which builds its tables in the same launch.  By-distance modes write the
// value into each reversed copy, and the thread with x < k also writes the
// zero that pads position x of copy k.
__device__ __forceinline__ void table_entry(const TableArgs& a, int h, int x) {
  const float alpha = a.alpha[h], beta = a.beta[h], mu = a.mu[h];
  float b, g1, g2;
  if (a.mode == kTableDecode) {
    float val = 0.0f;
    if (x < a.Tkv) {
      bias_terms<false>(a.Tkv - 1 - x, alpha, beta, mu, a.eps, a.prior, &b, &g1, &g2);
      val = to_f32_finite(b * static_cast<float>(kLog2e));
    }
    a.tab[static_cast<size_t>(h) * a.len + x] = val;
    return;
  }
  const int nplanes = a.mode == kTableBackward ? 3 : 1;
  g1 = g2 = 0.0f;
  if (nplanes == 3)
    bias_terms<true>(x - a.off, alpha, beta, mu, a.eps, a.prior, &b, &g1, &g2);
  else
    bias_terms<false>(x - a.off, alpha, beta, mu, a.eps, a.prior, &b, &g1, &g2);
  const float val[3] = {to_f32_finite(b * static_cast<float>(kLog2e)), to_f32_finite(g1),
                        to_f32_finite(g2)};
  const size_t row = static_cast<size_t>(a.len);
  const size_t plane = static_cast<size_t>(kTabCopies) * a.H * row;
  for (int p = 0; p < nplanes; ++p) {
#pragma unroll
    for (int k = 0; k < kTabCopies; ++k) {
      float* dst = a.tab + p * plane + (static_cast<size_t>(k) * a.H + h) * row;
      if (x >= k) dst[a.len - 1 - x + k] = val[p];
      if (x < k) dst[x] = 0.0f;
    }
  }
}

}  // namespace bam
