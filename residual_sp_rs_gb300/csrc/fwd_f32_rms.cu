// Forward instances: activation f32, norm rms.
#include "fwd_inst.cuh"

namespace spf {
cudaError_t launch_fwd_f32_rms(const FwdArgs& a, int T, const RowShape& s, dim3 grid,
                                  cudaStream_t st) {
  return launch_fwd_impl<float, false>(a, T, s, grid, st);
}
}  // namespace spf
