// bwd_tma.cu -- launch of the TMA-fed backward (bf16, H a multiple of 16).
#include "bwd_tma.cuh"
#include "launch.h"

namespace spf {

namespace {

template <bool LN>
void (*tma_kernel(int vpt))(const BwdArgs, const BwdTmaLayout) {
  switch (vpt) {
    case 1: return sp_bwd_tma_kernel<LN, 1>;
    case 2: return sp_bwd_tma_kernel<LN, 2>;
    case 3: return sp_bwd_tma_kernel<LN, 3>;
    case 4: return sp_bwd_tma_kernel<LN, 4>;
    default: return nullptr;
  }
}

constexpr size_t kStaticSmem = 1024;  // the kernel's static shared arrays, rounded up

}  // namespace

bool plan_bwd_tma(int64_t H, bool ln, bool has_dh, bool has_mask, int max_smem, BwdTmaPlan* p) {
  if (H % 16 != 0) return false;  // mask rows must be whole 16-byte copies
  const int nvec = (int)(H / 8);
  int tpr = 32;
  while (tpr < 256 && (nvec + tpr - 1) / tpr > 4) tpr *= 2;
  const int vpt = (nvec + tpr - 1) / tpr;
  if (vpt > 4) return false;
  const int nrg = tpr >= 256 ? 1 : 256 / tpr;
  const uint32_t rowb = (uint32_t)H * 2;
  BwdTmaLayout L = {};
  L.off_h = rowb;
  L.off_dh = 2 * rowb;
  L.off_mask = has_dh ? 3 * rowb : 2 * rowb;
  L.stage_bytes = L.off_mask + (has_mask ? (uint32_t)H : 0u);
  L.stage_bytes = (L.stage_bytes + 15u) & ~15u;
  L.row_tx = 2 * rowb + (has_dh ? rowb : 0u) + (has_mask ? (uint32_t)H : 0u);
  L.nrg = nrg;
  const size_t fixed_base = (size_t)(ln ? 2 : 1) * H * 4 + (size_t)nvec * 16;
  const size_t budget = (size_t)max_smem - kStaticSmem;
  int nst = 0;
  // stages, rounded down to a multiple of the row groups (each owns its stages)
  for (int cand = 64; cand >= 2 * nrg; --cand) {
    if (cand % nrg) continue;
    const size_t bars = 16 * (((size_t)2 * cand * 8 + 15) / 16);
    if (bars + fixed_base + (size_t)cand * L.stage_bytes <= budget) {
      nst = cand;
      break;
    }
  }
  if (nst < 2 * nrg) return false;
  L.nst = nst;
  L.smem_stages = (uint32_t)(16 * (((size_t)2 * nst * 8 + 15) / 16) + fixed_base);
  p->layout = L;
  p->shape.tpr = tpr;
  p->shape.vpt = vpt;
  p->shape.block = nrg * tpr + 32;
  p->smem = L.smem_stages + (size_t)nst * L.stage_bytes;
  return true;
}

cudaError_t launch_bwd_tma(bool ln, const BwdArgs& a, const BwdTmaPlan& p, dim3 grid,
                           cudaStream_t st) {
  void (*k)(const BwdArgs, const BwdTmaLayout) = ln ? tma_kernel<true>(p.shape.vpt)
                                                    : tma_kernel<false>(p.shape.vpt);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  return pdl_launch(k, grid, dim3(p.shape.block), p.smem, st, a, p.layout);
}

}  // namespace spf
