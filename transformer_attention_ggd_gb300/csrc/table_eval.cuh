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
__device__ __forceinline__ void bias_terms(int dint, float alpha, float beta, float mu, float eps,
                                           float* b, float* dbeta, float* dmu) {
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
  *dbeta = bb * ((fe + lm) * 0.69314718055994530942f);  // b ln r
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
      bias_terms(a.Tkv - 1 - x, alpha, beta, mu, a.eps, &b, &g1, &g2);
      val = to_f32_finite(b * static_cast<float>(kLog2e));
    }
    a.tab[static_cast<size_t>(h) * a.len + x] = val;
    return;
  }
  bias_terms(x - a.off, alpha, beta, mu, a.eps, &b, &g1, &g2);
  const float val[3] = {to_f32_finite(b * static_cast<float>(kLog2e)), to_f32_finite(g1),
                        to_f32_finite(g2)};
  const int nplanes = a.mode == kTableBackward ? 3 : 1;
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
