// TMA-fed backward instances: bf16, norm ln.
#include "bwd_tma_inst.cuh"

namespace spf {
cudaError_t launch_bwd_tma_ln(const BwdArgs& a, const BwdTmaPlan& p, dim3 grid, cudaStream_t st) {
  return launch_bwd_tma_impl<true>(a, p, grid, st);
}
}  // namespace spf
