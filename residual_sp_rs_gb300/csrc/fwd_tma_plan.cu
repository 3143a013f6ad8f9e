// fwd_tma_plan.cu -- shape of the TMA-fed forward's shared-memory ring.
#include "launch.h"

namespace spf {

namespace {
constexpr size_t kStaticSmem = 1024;  // the kernel's static shared arrays, rounded up
constexpr int kMaxConsumers = 512;
}  // namespace

// Picks the row-group width (<= 3 vectors per thread) and rows per stage that
// give the most consumer threads while at least two stages fit in shared
// memory next to gamma/beta; false when no such ring exists (long rows).
bool plan_fwd_tma(int64_t H, int T, bool ln, int max_smem, int64_t rows, int sms, FwdTmaPlan* p) {
  const int nvec = (int)(H / 8);
  const size_t rowb = (size_t)H * 2;
  const size_t gb = (size_t)H * 4 * (ln ? 2 : 1);
  const size_t budget = (size_t)max_smem - kStaticSmem;
  bool found = false;
  int best_threads = 0;
  for (int tpr = 32; tpr <= kMaxConsumers; tpr *= 2) {
    const int vpt = (nvec + tpr - 1) / tpr;
    if (vpt > 3) continue;
    for (int nrg = kMaxConsumers / tpr; nrg >= 1; nrg /= 2) {
      if (tpr > 32 && nrg > 15) continue;  // named barriers 1..nrg
      const size_t blk = (size_t)nrg * rowb;
      const size_t stage = blk * (size_t)(T + 1);
      int nst = 0;
      for (int cand = 4; cand >= 2; --cand) {
        const size_t bars = 16 * (((size_t)2 * cand * 8 + 15) / 16);
        if (bars + gb + (size_t)cand * stage <= budget) {
          nst = cand;
          break;
        }
      }
      if (nst < 2) continue;
      if (nrg * tpr > best_threads) {
        best_threads = nrg * tpr;
        found = true;
        FwdTmaLayout L = {};
        L.nst = nst;
        L.nrg = nrg;
        L.stage_bytes = (uint32_t)stage;
        L.blk = (uint32_t)blk;
        L.smem_stages = (uint32_t)(16 * (((size_t)2 * nst * 8 + 15) / 16) + gb);
        const int64_t ctas = rows < sms ? (rows > 0 ? rows : 1) : sms;
        L.rows_per_cta = rows > 0 ? (rows + ctas - 1) / ctas : 1;
        p->layout = L;
        p->shape.tpr = tpr;
        p->shape.vpt = vpt;
        p->shape.block = nrg * tpr + 32;
        p->smem = L.smem_stages + (size_t)nst * stage;
      }
      break;  // the largest fitting nrg for this width
    }
  }
  return found;
}

}  // namespace spf
