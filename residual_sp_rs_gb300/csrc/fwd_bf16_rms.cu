// Forward instances: activation bf16, norm rms.
#include "fwd_inst.cuh"

namespace spf {
cudaError_t launch_fwd_bf16_rms(const FwdArgs& a, int T, const RowShape& s, dim3 grid,
                                  cudaStream_t st) {
  return launch_fwd_impl<__nv_bfloat16, false>(a, T, s, grid, st);
}
}  // namespace spf
