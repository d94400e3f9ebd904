// Evaluation of one entry of the per-head distance tables (see table.cu),
// shared by the table kernel and the backward preprocess.
#pragma once

#include "bam_common.cuh"

namespace bam {

// b, db/dbeta and db/dmu at distance d.  fp32 arithmetic except for the
// exponent y = beta * log2(u / alpha), which is assembled in double from the
// exact binary exponent of u/alpha and an fp32 log2 of its mantissa (absolute
// error ~1e-7); 2^y is then an exact power of two times exp2f of the
// fractional part.  The relative error of b is a few 1e-7 whatever its
// magnitude, where a plain fp32 pow loses ~1e-7 * |y| (1e-6 at |b| ~ 1e4).
// The few double operations per entry keep the table cheap on a GPU whose
// fp64 rate is low.
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
  const float mant = frexpf(r, &e2);                               // r = mant * 2^e2
  const double L = static_cast<double>(e2) + static_cast<double>(log2f(mant));  // log2(r)
  double y = static_cast<double>(beta) * L;
  y = fmin(fmax(y, -400.0), 400.0);
  const double n = floor(y);
  const float pw = ldexpf(exp2f(static_cast<float>(y - n)), static_cast<int>(n));  // 2^y
  const float bb = -pw;
  *b = bb;
  *dbeta = static_cast<float>(static_cast<double>(bb) * L * 0.69314718055994530942);  // b ln r
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
// which builds its tables in the same launch.
__device__ __forceinline__ void table_entry(const TableArgs& a, int h, int x) {
  const float alpha = a.alpha[h], beta = a.beta[h], mu = a.mu[h];
  const size_t idx = static_cast<size_t>(h) * a.len + x;
  float b, g1, g2;
  if (a.mode == kTableDecode) {
    float val = 0.0f;
    if (x < a.Tkv) {
      bias_terms(a.Tkv - 1 - x, alpha, beta, mu, a.eps, &b, &g1, &g2);
      val = to_f32_finite(b * static_cast<float>(kLog2e));
    }
    a.tab[idx] = val;
    return;
  }
  bias_terms(x - a.off, alpha, beta, mu, a.eps, &b, &g1, &g2);
  a.tab[idx] = to_f32_finite(b * static_cast<float>(kLog2e));
  if (a.mode == kTableBackward) {
    const size_t plane = static_cast<size_t>(a.H) * a.len;
    a.tab[plane + idx] = to_f32_finite(g1);
    a.tab[2 * plane + idx] = to_f32_finite(g2);
  }
}

}  // namespace bam
