// bwd_tma_inst.cuh -- instances of the TMA-fed backward for one norm:
// VPT (1..4 RMSNorm, 1..2 LayerNorm), dh_out present or not, mask mode, and
// the two block sizes (544 threads for VPT <= 3).
#pragma once

#include "bwd_tma.cuh"
#include "launch.h"

namespace spf {

using BwdTmaKernel = void (*)(const BwdArgs, const BwdTmaLayout);

template <bool LN, bool DH, bool MASK, bool REGEN, int NTHR>
BwdTmaKernel bwd_tma_kernel_v(int vpt) {
  switch (vpt) {
    case 1: return sp_bwd_tma_kernel<LN, 1, DH, MASK, REGEN, NTHR>;
    case 2: return sp_bwd_tma_kernel<LN, 2, DH, MASK, REGEN, NTHR>;
    case 3:
      if constexpr (!LN) return sp_bwd_tma_kernel<LN, 3, DH, MASK, REGEN, NTHR>;  // LayerNorm stays <= 2
      return nullptr;
    case 4:
      if constexpr (!LN && NTHR == kBwdTmaNarrow) return sp_bwd_tma_kernel<LN, 4, DH, MASK, REGEN, NTHR>;
      return nullptr;
    default: return nullptr;
  }
}

// mode: 0 = no dropout, 1 = stored mask, 2 = regenerate the mask
template <bool LN, int NTHR>
BwdTmaKernel bwd_tma_kernel_m(int vpt, bool dh, int mode) {
  if (dh) {
    if (mode == 1) return bwd_tma_kernel_v<LN, true, true, false, NTHR>(vpt);
    if (mode == 2) return bwd_tma_kernel_v<LN, true, false, true, NTHR>(vpt);
    return bwd_tma_kernel_v<LN, true, false, false, NTHR>(vpt);
  }
  if (mode == 1) return bwd_tma_kernel_v<LN, false, true, false, NTHR>(vpt);
  if (mode == 2) return bwd_tma_kernel_v<LN, false, false, true, NTHR>(vpt);
  return bwd_tma_kernel_v<LN, false, false, false, NTHR>(vpt);
}

template <bool LN>
cudaError_t launch_bwd_tma_impl(const BwdArgs& a, const BwdTmaPlan& p, dim3 grid, cudaStream_t st) {
  const bool dh = a.dh != nullptr;
  const int mode = a.mask ? 1 : (a.regen ? 2 : 0);
  const BwdTmaKernel k = p.nthr == kBwdTmaMid ? bwd_tma_kernel_m<LN, kBwdTmaMid>(p.shape.vpt, dh, mode)
                                              : bwd_tma_kernel_m<LN, kBwdTmaNarrow>(p.shape.vpt, dh, mode);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  return pdl_launch(k, grid, dim3(p.shape.block), p.smem, st, a, p.layout);
}

}  // namespace spf
