// bwd_tma.cu -- launch of the TMA-fed backward (bf16, H a multiple of 16).
#include "bwd_tma.cuh"
#include "launch.h"

namespace spf {

namespace {

template <bool LN, bool DH, bool MASK, bool REGEN>
void (*tma_kernel_v(int vpt))(const BwdArgs, const BwdTmaLayout) {
  switch (vpt) {
    case 1: return sp_bwd_tma_kernel<LN, 1, DH, MASK, REGEN>;
    case 2: return sp_bwd_tma_kernel<LN, 2, DH, MASK, REGEN>;
    case 3:
      if constexpr (!LN) return sp_bwd_tma_kernel<LN, 3, DH, MASK, REGEN>;  // LayerNorm stays <= 2
      return nullptr;
    case 4:
      if constexpr (!LN) return sp_bwd_tma_kernel<LN, 4, DH, MASK, REGEN>;
      return nullptr;
    default: return nullptr;
  }
}

// mode: 0 = no dropout, 1 = stored mask, 2 = regenerate the mask
template <bool LN>
void (*tma_kernel(int vpt, bool dh, int mode))(const BwdArgs, const BwdTmaLayout) {
  if (dh) {
    if (mode == 1) return tma_kernel_v<LN, true, true, false>(vpt);
    if (mode == 2) return tma_kernel_v<LN, true, false, true>(vpt);
    return tma_kernel_v<LN, true, false, false>(vpt);
  }
  if (mode == 1) return tma_kernel_v<LN, false, true, false>(vpt);
  if (mode == 2) return tma_kernel_v<LN, false, false, true>(vpt);
  return tma_kernel_v<LN, false, false, false>(vpt);
}

constexpr size_t kStaticSmem = 1024;  // the kernel's static shared arrays, rounded up
constexpr int kBwdTmaConsumers = 480;  // consumer threads per CTA (+1 producer warp: 16 warps)

}  // namespace

bool plan_bwd_tma(int64_t H, bool ln, bool has_dh, bool has_mask, int max_smem, BwdTmaPlan* p) {
  if (H % 16 != 0) return false;  // mask rows must be whole 16-byte copies
  const int nvec = (int)(H / 8);
  // up to 15 consumer warps; a row group of tpr (<= 256) threads holds <= 4
  // vectors per thread (<= 2 for LayerNorm, whose dbeta accumulators add
  // registers)
  const int vcap = ln ? 2 : 4;
  int tpr = 32;
  while (tpr < 256 && (nvec + tpr - 1) / tpr > vcap) tpr *= 2;
  const int vpt = (nvec + tpr - 1) / tpr;
  if (vpt > vcap) return false;
  int nrg = kBwdTmaConsumers / tpr;  // rows per stage, one per row group
  const uint32_t rowb = (uint32_t)H * 2;
  const size_t fixed_base = (size_t)H * 4;  // gamma, fp32
  const size_t budget = (size_t)max_smem - kStaticSmem;
  for (; nrg >= 1; nrg /= 2) {
    BwdTmaLayout L = {};
    const uint32_t blk = (uint32_t)nrg * rowb;  // one tensor's rows in a stage
    L.off_h = blk;
    L.off_dh = 2 * blk;
    L.off_mask = has_dh ? 3 * blk : 2 * blk;
    L.stage_bytes = (L.off_mask + (has_mask ? (uint32_t)(nrg * H) : 0u) + 15u) & ~15u;
    L.nrg = nrg;
    int nst = 0;
    for (int cand = 8; cand >= 2; --cand) {
      const size_t bars = 16 * (((size_t)2 * cand * 8 + 15) / 16);
      if (bars + fixed_base + (size_t)cand * L.stage_bytes <= budget) {
        nst = cand;
        break;
      }
    }
    if (nst < 2) continue;  // fewer rows per stage, and try again
    // at the end the ring holds the row groups' column sums
    if ((size_t)nst * L.stage_bytes < (size_t)nrg * (ln ? 2 : 1) * H * 4) continue;
    // row groups wider than a warp synchronise on named barriers 1..nrg
    if (tpr > 32 && nrg > 15) return false;
    L.nst = nst;
    L.smem_stages = (uint32_t)(16 * (((size_t)2 * nst * 8 + 15) / 16) + fixed_base);
    p->layout = L;
    p->shape.tpr = tpr;
    p->shape.vpt = vpt;
    p->shape.block = nrg * tpr + 32;
    p->smem = L.smem_stages + (size_t)nst * L.stage_bytes;
    return true;
  }
  return false;
}

cudaError_t launch_bwd_tma(bool ln, const BwdArgs& a, const BwdTmaPlan& p, dim3 grid,
                           cudaStream_t st) {
  const bool dh = a.dh != nullptr;
  const int mode = a.mask ? 1 : (a.regen ? 2 : 0);
  void (*k)(const BwdArgs, const BwdTmaLayout) = ln ? tma_kernel<true>(p.shape.vpt, dh, mode)
                                                    : tma_kernel<false>(p.shape.vpt, dh, mode);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  return pdl_launch(k, grid, dim3(p.shape.block), p.smem, st, a, p.layout);
}

}  // namespace spf
