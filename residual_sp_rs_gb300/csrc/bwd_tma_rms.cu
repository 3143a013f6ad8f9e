// TMA-fed backward instances: bf16, norm rms.
#include "bwd_tma_inst.cuh"

namespace spf {
cudaError_t launch_bwd_tma_rms(const BwdArgs& a, const BwdTmaPlan& p, dim3 grid, cudaStream_t st) {
  return launch_bwd_tma_impl<false>(a, p, grid, st);
}
}  // namespace spf
