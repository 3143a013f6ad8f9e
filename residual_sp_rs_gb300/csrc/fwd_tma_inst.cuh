// fwd_tma_inst.cuh -- instances of the TMA-fed forward for one norm over
// T = 1..8, VPT = 1..3, the fast / generic rounding mode, the two block
// sizes (the 896-thread one only for T <= 4) and whole-row or column-chunk
// stages (one translation unit each).
#pragma once

#include "fwd_tma.cuh"
#include "launch.h"

namespace spf {

// CH (column chunks) only with 2 or 3 vectors per thread: one vector slot is
// a whole row.
template <bool LN, int T, bool FAST, int NTHR, bool CH>
inline void (*fwd_tma_kernel_for_vpt(int vpt))(const FwdArgs, const FwdTmaLayout) {
  switch (vpt) {
    case 1:
      if constexpr (!CH) return sp_fwd_tma_kernel<T, LN, 1, FAST, NTHR, false>;
      return nullptr;
    case 2: return sp_fwd_tma_kernel<T, LN, 2, FAST, NTHR, CH>;
    case 3: return sp_fwd_tma_kernel<T, LN, 3, FAST, NTHR, CH>;
    default: return nullptr;
  }
}

template <bool LN, int T, int NTHR, bool CH>
inline void (*fwd_tma_kernel_for_mode(int vpt, bool fast))(const FwdArgs, const FwdTmaLayout) {
  return fast ? fwd_tma_kernel_for_vpt<LN, T, true, NTHR, CH>(vpt)
              : fwd_tma_kernel_for_vpt<LN, T, false, NTHR, CH>(vpt);
}

template <bool LN, int T, bool CH>
inline void (*fwd_tma_kernel_for(int vpt, bool fast, int nthr))(const FwdArgs, const FwdTmaLayout) {
  if (nthr == kFwdTmaWide) {
    if constexpr (T <= kFwdTmaWideMaxT) return fwd_tma_kernel_for_mode<LN, T, kFwdTmaWide, CH>(vpt, fast);
    return nullptr;
  }
  return fwd_tma_kernel_for_mode<LN, T, kFwdTmaDeep, CH>(vpt, fast);
}

template <bool LN, bool CH>
cudaError_t launch_fwd_tma_impl(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid,
                                cudaStream_t st) {
  void (*k)(const FwdArgs, const FwdTmaLayout) = nullptr;
  const bool fast = a.dropout && !a.dyadic_scale;
  switch (T) {
    case 1: k = fwd_tma_kernel_for<LN, 1, CH>(p.shape.vpt, fast, p.nthr); break;
    case 2: k = fwd_tma_kernel_for<LN, 2, CH>(p.shape.vpt, fast, p.nthr); break;
    case 3: k = fwd_tma_kernel_for<LN, 3, CH>(p.shape.vpt, fast, p.nthr); break;
    case 4: k = fwd_tma_kernel_for<LN, 4, CH>(p.shape.vpt, fast, p.nthr); break;
    case 5: k = fwd_tma_kernel_for<LN, 5, CH>(p.shape.vpt, fast, p.nthr); break;
    case 6: k = fwd_tma_kernel_for<LN, 6, CH>(p.shape.vpt, fast, p.nthr); break;
    case 7: k = fwd_tma_kernel_for<LN, 7, CH>(p.shape.vpt, fast, p.nthr); break;
    case 8: k = fwd_tma_kernel_for<LN, 8, CH>(p.shape.vpt, fast, p.nthr); break;
    default: break;
  }
  if (!k) return cudaErrorInvalidValue;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  return pdl_launch(k, grid, dim3(p.shape.block), p.smem, st, a, p.layout);
}

}  // namespace spf
