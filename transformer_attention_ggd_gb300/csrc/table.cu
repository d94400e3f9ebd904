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
// Values are computed in fp32 with an error-compensated exponent (see
// table_eval.cuh) and stored pre-multiplied by log2(e) so that the softmax
// can run on exp2.  The backward mode also writes
// db/dbeta and db/dmu (natural units):
//   db/dbeta = b * ln(u / alpha)
//   db/dmu   = -beta * b * sgn(d - mu) / u      (0 inside the eps clamp)
// and 0 for both at u = 0.  db/dalpha = -beta * b / alpha needs no table.
#include "table_eval.cuh"

namespace bam {
namespace {

__global__ void bam_table_kernel(const TableArgs a) {
  // Let the next kernel of this call start its prologue.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // First kernel of every call that builds a table: the call starts here.
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) status_begin_call(a.status);
  const int h = blockIdx.y;
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= a.H || x >= a.len) return;
  table_entry(a, h, x);
}

}  // namespace

cudaError_t launch_table(const TableArgs& a, cudaStream_t st) {
  dim3 grid((a.len + 255) / 256, a.H);
  return launch_k(bam_table_kernel, grid, dim3(256), 0, st, false, a);
}

}  // namespace bam
