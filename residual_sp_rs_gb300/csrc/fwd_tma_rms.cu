// TMA-fed forward instances: bf16, norm rms.
#include "fwd_tma_inst.cuh"

namespace spf {
cudaError_t launch_fwd_tma_rms(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid,
                                cudaStream_t st) {
  return launch_fwd_tma_impl<false>(a, T, p, grid, st);
}
}  // namespace spf
