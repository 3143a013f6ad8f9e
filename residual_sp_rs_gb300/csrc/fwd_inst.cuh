// fwd_inst.cuh -- instantiates the forward kernel for one (activation, norm)
// pair over T = 1..8 and VPT = 1..4 and picks the instance at run time.
#pragma once

#include "fwd.cuh"
#include "launch.h"

namespace spf {

template <typename Act, bool LN, int T>
inline void (*fwd_kernel_for_vpt(int vpt))(const FwdArgs) {
  switch (vpt) {
    case 1: return sp_fwd_kernel<Act, T, LN, 1>;
    case 2: return sp_fwd_kernel<Act, T, LN, 2>;
    case 3: return sp_fwd_kernel<Act, T, LN, 3>;
    case 4: return sp_fwd_kernel<Act, T, LN, 4>;
    default: return nullptr;
  }
}

template <typename Act, bool LN>
cudaError_t launch_fwd_impl(const FwdArgs& a, int T, const RowShape& s, dim3 grid,
                            cudaStream_t st) {
  void (*k)(const FwdArgs) = nullptr;
  switch (T) {
    case 1: k = fwd_kernel_for_vpt<Act, LN, 1>(s.vpt); break;
    case 2: k = fwd_kernel_for_vpt<Act, LN, 2>(s.vpt); break;
    case 3: k = fwd_kernel_for_vpt<Act, LN, 3>(s.vpt); break;
    case 4: k = fwd_kernel_for_vpt<Act, LN, 4>(s.vpt); break;
    case 5: k = fwd_kernel_for_vpt<Act, LN, 5>(s.vpt); break;
    case 6: k = fwd_kernel_for_vpt<Act, LN, 6>(s.vpt); break;
    case 7: k = fwd_kernel_for_vpt<Act, LN, 7>(s.vpt); break;
    case 8: k = fwd_kernel_for_vpt<Act, LN, 8>(s.vpt); break;
    default: break;
  }
  if (!k) return cudaErrorInvalidValue;
  const size_t smem = (size_t)a.nvec * 16 * (LN ? 2 : 1);  // gamma (+ beta) vectors
  if (smem > kSmemOptInThreshold) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return pdl_launch(k, grid, dim3(s.block), smem, st, a);
}

}  // namespace spf
