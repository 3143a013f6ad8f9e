// bwd_tma.cu -- shape of the TMA-fed backward's ring (bf16, H a multiple of
// 16) and its launch.
#include "launch.h"

namespace spf {

namespace {

constexpr size_t kStaticSmem = 1024;  // the kernel's static shared arrays, rounded up
constexpr int kMaxStages = 32;
// smallest bulk copy worth issuing: a stage takes enough rows that its dy
// copy moves at least this many bytes (up to one row per group)
constexpr size_t kMinCopy = 16384;

}  // namespace

// The narrowest row group (<= 4 vectors per thread, <= 2 for LayerNorm,
// whose dbeta accumulators add registers); as many row groups as the block
// allows (15 warps at 512 threads; when that leaves one row group of 8 warps
// and VPT <= 3, two in the 544-thread block, which re-reads dy and h from
// shared memory in the second pass) but no more than the rows a CTA owns;
// stages of rb rows, as many as fit next to gamma.
// At the end the ring must hold every row group's column sums.
bool plan_bwd_tma(int64_t H, bool ln, bool has_dh, bool has_mask, int max_smem, int64_t rows_per_cta,
                  BwdTmaPlan* p) {
  if (H % 16 != 0) return false;  // mask rows must be whole 16-byte copies
  const int nvec = (int)(H / 8);
  const int vcap = ln ? 2 : 4;
  int tpr = 32;
  while (tpr < 256 && (nvec + tpr - 1) / tpr > vcap) tpr *= 2;
  const int vpt = (nvec + tpr - 1) / tpr;
  if (vpt > vcap) return false;
  auto groups = [&](int block) {
    int g = (block / 32 - 1) / (tpr / 32);
    if (tpr > 32 && g > 15) g = 15;  // named barriers 1..g
    if ((int64_t)g > rows_per_cta) g = rows_per_cta > 0 ? (int)rows_per_cta : 1;
    return g;
  };
  // the narrow block keeps dy and xhat in registers between the passes,
  // which pays more than extra warps unless it leaves a single row group
  int nrg = groups(kBwdTmaNarrow);
  if (vpt <= 3 && nrg < 2 && groups(kBwdTmaMid) > nrg)
    nrg = groups(kBwdTmaMid);
  const int ns = ln ? 2 : 1;
  const uint32_t rowb = (uint32_t)H * 2;
  const size_t fixed_base = (size_t)H * 4;  // gamma, fp32
  if (max_smem <= (int)kStaticSmem) return false;  // no room for a ring at all
  const size_t budget = (size_t)max_smem - kStaticSmem;
  for (; nrg >= 1; --nrg) {
    const bool narrow = nrg * tpr + 32 <= kBwdTmaNarrow;
    int rb = (int)((kMinCopy + rowb - 1) / rowb);
    rb = rb < 1 ? 1 : (rb > nrg ? nrg : rb);
    // the narrow kernel needs rb to divide nrg (whole stages per round of rows)
    if (narrow)
      while (nrg % rb != 0) ++rb;
    for (; rb >= 1; --rb) {
      if (narrow && nrg % rb != 0) continue;
      BwdTmaLayout L = {};
      const uint32_t blk = (uint32_t)rb * rowb;  // one tensor's rows in a stage
      L.off_h = blk;
      L.off_dh = 2 * blk;
      L.off_mask = has_dh ? 3 * blk : 2 * blk;
      L.stage_bytes = (L.off_mask + (has_mask ? (uint32_t)(rb * H) : 0u) + 15u) & ~15u;
      L.nrg = nrg;
      L.rb = rb;
      // A row group waits for a stage by the parity of its ring slot's full
      // barrier, which is only unambiguous when the slot's previous stage
      // has landed.  So when slots are reused, every stage a group consumes
      // must come back to a slot whose previous stage the same group
      // consumed: the stages form `lanes` interleaved sequences (stage j to
      // the groups of lane j % lanes; rows go to the groups round robin),
      // and the ring holds a multiple of `lanes` stages.
      int lanes = nrg, g = rb;
      for (int a0 = nrg; g != 0;) {  // lanes = nrg / gcd(nrg, rb)
        const int t = a0 % g;
        a0 = g;
        g = t;
        if (g == 0) lanes = nrg / a0;
      }
      const int64_t nstage = (rows_per_cta + rb - 1) / rb;
      int nst = 0;
      for (int cand = kMaxStages; cand >= 2; --cand) {
        const size_t bars = 16 * (((size_t)2 * cand * 8 + 15) / 16);
        const bool reuse = nstage > cand;
        if ((!reuse || cand % lanes == 0) && bars + fixed_base + (size_t)cand * L.stage_bytes <= budget) {
          nst = cand;
          break;
        }
      }
      if (nst < 2) continue;  // fewer rows per stage
      // at the end the ring holds the row groups' column sums
      if ((size_t)nst * L.stage_bytes < (size_t)nrg * ns * 8 * (nvec + 4) * 4) continue;
      L.nst = nst;
      L.pf_stages = prefetch_stages(L.stage_bytes);
      L.smem_stages = (uint32_t)(16 * (((size_t)2 * nst * 8 + 15) / 16) + fixed_base);
      p->layout = L;
      p->shape.tpr = tpr;
      p->shape.vpt = vpt;
      p->shape.block = nrg * tpr + 32;
      p->nthr = p->shape.block <= kBwdTmaNarrow ? kBwdTmaNarrow : kBwdTmaMid;
      p->smem = L.smem_stages + (size_t)nst * L.stage_bytes;
      return true;
    }
  }
  return false;
}

cudaError_t launch_bwd_tma(bool ln, const BwdArgs& a, const BwdTmaPlan& p, dim3 grid,
                           cudaStream_t st) {
  return ln ? launch_bwd_tma_ln(a, p, grid, st) : launch_bwd_tma_rms(a, p, grid, st);
}

}  // namespace spf
