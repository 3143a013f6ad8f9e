// bwd.cu -- backward instances (activation x norm x VPT) and launchers.
#include "bwd.cuh"
#include "launch.h"

namespace spf {

namespace {

template <typename Act, bool LN>
void (*bwd_kernel_for(int vpt))(const BwdArgs) {
  switch (vpt) {
    case 1: return sp_bwd_kernel<Act, LN, 1>;
    case 2: return sp_bwd_kernel<Act, LN, 2>;
    case 3: return sp_bwd_kernel<Act, LN, 3>;
    case 4: return sp_bwd_kernel<Act, LN, 4>;
    default: return nullptr;
  }
}

void (*bwd_kernel(int dtype, bool ln, int vpt))(const BwdArgs) {
  if (dtype == 1) return ln ? bwd_kernel_for<__nv_bfloat16, true>(vpt) : bwd_kernel_for<__nv_bfloat16, false>(vpt);
  return ln ? bwd_kernel_for<float, true>(vpt) : bwd_kernel_for<float, false>(vpt);
}

}  // namespace

// How many 8-CTA clusters of the backward kernel can be resident at once on
// the current device (clusters must fit inside one GPC, so this is at most,
// and often below, SMs * CTAs-per-SM / 8).
int bwd_max_active_clusters(int dtype, bool ln, const RowShape& s, size_t smem) {
  void (*k)(const BwdArgs) = bwd_kernel(dtype, ln, s.vpt);
  if (!k) return 0;
  if (smem > kSmemOptInThreshold &&
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kBwdCluster * 64);
  cfg.blockDim = dim3(s.block);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)k, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_bwd(int dtype, bool ln, const BwdArgs& a, const RowShape& s, dim3 grid,
                       size_t smem, cudaStream_t st) {
  void (*k)(const BwdArgs) = bwd_kernel(dtype, ln, s.vpt);
  if (!k) return cudaErrorInvalidValue;
  if (smem > kSmemOptInThreshold) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return pdl_launch(k, grid, dim3(s.block), smem, st, a);
}

cudaError_t launch_colsum(const float* ws, int nparts, int H, bool ln, float* dgamma,
                          float* dbeta, bool accumulate, cudaStream_t st) {
  const int n4 = H / 4;
  const dim3 grid((unsigned)((n4 + 31) / 32), ln ? 2u : 1u);
  return pdl_launch(sp_colsum_kernel, grid, dim3(32, 32), 0, st, ws, nparts, H, dgamma, dbeta,
                    accumulate ? 1 : 0);
}

}  // namespace spf
