// TMA-fed forward instances: bf16, norm rms, column-chunk stages.
#include "fwd_tma_inst.cuh"

namespace spf {
cudaError_t launch_fwd_tma_rms_ch(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid,
                                   cudaStream_t st) {
  return launch_fwd_tma_impl<false, true>(a, T, p, grid, st);
}
}  // namespace spf
