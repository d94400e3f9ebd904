// Self-test of the failure detection: one thread waits, through the same
// bounded mbarrier wait every kernel of the library uses, on a barrier that
// nothing ever arrives at.  After the wall-clock limit the wait gives up,
// records BAM_ERR_TIMEOUT (site kSiteSelftest) in the workspace status word
// and the kernel returns, so the context stays usable and
// bam_attn_check_status reports the give-up.  No trap, no fault, no hang.
#include "../../include/bam_attn.h"
#include "bam_common.cuh"

namespace bam {
namespace {

constexpr int kSiteSelftest = 90;

__global__ void bam_selftest_wait_kernel(DevStatus* st) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    status_begin_call(st);
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Phase 0 of a barrier that expects one arrival and gets none never
  // completes: the wait runs into its limit.
  if (threadIdx.x == 0) mbar_wait(&bar, 0, st, &abort_flag, kSiteSelftest);
}

}  // namespace
}  // namespace bam

using namespace bam;

extern "C" bam_status bam_attn_selftest_wait(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < kStatusBytes)
    return BAM_ERR_WORKSPACE;
  DevStatus* st = static_cast<DevStatus*>(ws);
  bam_selftest_wait_kernel<<<1, 32, 0, stream>>>(st);
  return cudaGetLastError() == cudaSuccess ? BAM_OK : BAM_ERR_CUDA;
}
