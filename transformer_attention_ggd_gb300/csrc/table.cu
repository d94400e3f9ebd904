// Per-head relative-distance table of the GGD-BAM bias.
//
// b_h(d) = -(u / alpha_h)^beta_h with u = |d - mu_h|, clamped to max(u, eps)
// when beta_h <= 0 ("Bayesian Attention Mechanism" summary, "Solution
// Proposee : GGD-BAM"; eps from the BAM README, "Implementation Details").
// The bias depends on (h, d) only, so it is evaluated once per distance
// (H x O(T) power evaluations instead of one per query-key pair) and the
// attention kernels read it from shared memory.  Keeping a 1-D table per
// relative distance follows the Sandwich entry of the attention-gym
// "Score Mods" page.
//
// Values are computed in fp64 and stored in fp32, pre-multiplied by log2(e)
// so that the softmax can run on exp2.  The backward mode also writes
// db/dbeta and db/dmu (natural units):
//   db/dbeta = b * ln(u / alpha)
//   db/dmu   = -beta * b * sgn(d - mu) / u      (0 inside the eps clamp)
// and 0 for both at u = 0.  db/dalpha = -beta * b / alpha needs no table.
#include "bam_common.cuh"

namespace bam {

namespace {

__device__ __forceinline__ void bias_terms(double d, double alpha, double beta, double mu,
                                           double eps, double* b, double* dbeta,
                                           double* dmu) {
  double u = fabs(d - mu);
  bool clamped = false;
  if (beta <= 0.0 && u < eps) {
    u = eps;
    clamped = true;
  }
  if (u == 0.0) {
    *b = 0.0;
    *dbeta = 0.0;
    *dmu = 0.0;
    return;
  }
  const double r = u / alpha;
  const double bb = -pow(r, beta);
  *b = bb;
  *dbeta = bb * log(r);
  const double sgn = (d - mu > 0.0) ? 1.0 : -1.0;
  *dmu = clamped ? 0.0 : -beta * bb * sgn / u;
}

__device__ __forceinline__ float to_f32_finite(double x) {
  float f = static_cast<float>(x);
  // Keep the table finite so that exp2 of a difference never sees inf - inf.
  if (f < -3.0e38f) f = -3.0e38f;
  if (f > 3.0e38f) f = 3.0e38f;
  return f;
}

__global__ void bam_table_kernel(const TableArgs a) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 4) {
    reinterpret_cast<int*>(a.status)[threadIdx.x] = 0;
  }
  const int h = blockIdx.y;
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= a.H || x >= a.len) return;
  const double alpha = a.alpha[h], beta = a.beta[h], mu = a.mu[h];
  const size_t idx = static_cast<size_t>(h) * a.len + x;
  if (a.mode == kTableDecode) {
    float val = 0.0f;
    if (x < a.Tkv) {
      double b, g1, g2;
      bias_terms(static_cast<double>(a.Tkv - 1 - x), alpha, beta, mu, a.eps, &b, &g1, &g2);
      val = to_f32_finite(b * kLog2e);
    }
    a.tab[idx] = val;
    return;
  }
  double b, g1, g2;
  bias_terms(static_cast<double>(x - a.off), alpha, beta, mu, a.eps, &b, &g1, &g2);
  a.tab[idx] = to_f32_finite(b * kLog2e);
  if (a.mode == kTableBackward) {
    const size_t plane = static_cast<size_t>(a.H) * a.len;
    a.tab[plane + idx] = to_f32_finite(g1);
    a.tab[2 * plane + idx] = to_f32_finite(g2);
  }
}

}  // namespace

cudaError_t launch_table(const TableArgs& a, cudaStream_t st) {
  dim3 grid((a.len + 255) / 256, a.H);
  bam_table_kernel<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace bam
