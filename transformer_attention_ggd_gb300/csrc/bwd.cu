// Backward launchers (kernels follow).
#include "bam_common.cuh"

namespace bam {
cudaError_t launch_bwd_prep(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, const BwdArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_bwd_final(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace bam
