// TMA-fed forward instances: bf16, norm ln, column-chunk stages.
#include "fwd_tma_inst.cuh"

namespace spf {
cudaError_t launch_fwd_tma_ln_ch(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid,
                                   cudaStream_t st) {
  return launch_fwd_tma_impl<true, true>(a, T, p, grid, st);
}
}  // namespace spf
