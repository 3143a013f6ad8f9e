// fwd_tma_plan.cu -- shape of the TMA-fed forward's shared-memory ring.
#include "launch.h"

namespace spf {

namespace {
constexpr size_t kStaticSmem = 1024;  // the kernel's static shared arrays, rounded up
constexpr int kMaxStages = 48;
// smallest bulk copy worth issuing: a stage takes enough rows that each of
// its T+1 copies moves at least this many bytes (up to one row per group)
constexpr size_t kMinCopy = 8192;

// The most stages of `stage` bytes that fit next to gamma/beta.  A row group
// waits for a stage by the parity of its ring slot's full barrier, which is
// only unambiguous when the slot's previous stage has landed; so when the
// CTA's `nstage` stages reuse slots, the ring holds a multiple of `lanes`
// stages, which brings every slot back to the row group that consumed its
// previous stage.
int ring_stages(size_t stage, size_t gb, size_t budget, int64_t nstage, int lanes) {
  for (int cand = kMaxStages; cand >= 2; --cand) {
    const size_t bars = 16 * (((size_t)2 * cand * 8 + 15) / 16);
    if ((nstage <= cand || cand % lanes == 0) && bars + gb + (size_t)cand * stage <= budget) return cand;
  }
  return 0;
}

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}
}  // namespace

// Picks the narrowest row group (<= 3 vectors per thread), as many row groups
// as the block size allows but no more than the rows a CTA owns, and stages
// of rb rows (copies of at least kMinCopy bytes where the ring allows), as
// many as fit in shared memory next to gamma/beta (at least two).  When two
// one-row stages do not fit (T*H large), stages of one column chunk of a row;
// false when not even those fit.  T <= 4 takes the 896-thread
// block (more rows in flight per SM); larger T the 544-thread one, which
// leaves each thread more registers.
bool plan_fwd_tma(int64_t H, int T, bool ln, int max_smem, int64_t rows, int sms, FwdTmaPlan* p) {
  const int nvec = (int)(H / 8);
  const size_t rowb = (size_t)H * 2;
  const size_t gb = (size_t)H * 4 * (ln ? 2 : 1);
  if (max_smem <= (int)kStaticSmem) return false;  // no room for a ring at all
  const size_t budget = (size_t)max_smem - kStaticSmem;
  const int64_t ctas = rows < sms ? (rows > 0 ? rows : 1) : sms;
  const int64_t rows_per_cta = rows > 0 ? (rows + ctas - 1) / ctas : 1;
  const bool wide = T <= kFwdTmaWideMaxT;
  const int cons_warps = (wide ? kFwdTmaWide : kFwdTmaDeep) / 32 - 1;
  for (int tpr = 32; tpr / 32 <= cons_warps; tpr *= 2) {
    const int vpt = (nvec + tpr - 1) / tpr;
    if (vpt > 3) continue;
    int nrg = cons_warps / (tpr / 32);
    if (tpr > 32 && nrg > 15) nrg = 15;  // named barriers 1..nrg
    if ((int64_t)nrg > rows_per_cta) nrg = (int)rows_per_cta;
    int rb = (int)((kMinCopy + rowb - 1) / rowb);
    rb = rb < 1 ? 1 : (rb > nrg ? nrg : rb);
    // rows go to the row groups round robin: the groups of stage j recur
    // every nrg / gcd(nrg, rb) stages
    int nst = 0;
    for (; rb >= 1; --rb) {
      nst = ring_stages((size_t)rb * (T + 1) * rowb, gb, budget, (rows_per_cta + rb - 1) / rb,
                        nrg / gcd_int(nrg, rb));
      if (nst >= 2) break;
    }
    bool chunked = false;
    size_t blk = (size_t)rb * rowb, stage = blk * (T + 1);
    if (rb < 1) {
      // a whole row does not fit twice: stages of one column chunk (one
      // vector slot of the row group, tpr*16 bytes of each input)
      if (vpt < 2) return false;
      rb = 1;
      blk = (size_t)tpr * 16;
      stage = blk * (T + 1);
      // a row is vpt consecutive stages; row i belongs to group i % nrg (one
      // group consumes every stage in order: no constraint)
      nst = ring_stages(stage, gb, budget, rows_per_cta * vpt, nrg > 1 ? nrg * vpt : 1);
      if (nst < 2) return false;
      chunked = true;
    }
    FwdTmaLayout L = {};
    L.nst = nst;
    L.nrg = nrg;
    L.rb = rb;
    L.stage_bytes = (uint32_t)stage;
    L.blk = (uint32_t)blk;
    L.smem_stages = (uint32_t)(16 * (((size_t)2 * nst * 8 + 15) / 16) + gb);
    L.rows_per_cta = rows_per_cta;
    L.pf_stages = prefetch_stages(stage);
    p->layout = L;
    p->shape.tpr = tpr;
    p->shape.vpt = vpt;
    p->shape.block = nrg * tpr + 32;
    p->nthr = wide ? kFwdTmaWide : kFwdTmaDeep;
    p->chunked = chunked;
    p->smem = L.smem_stages + (size_t)nst * stage;
    return true;
  }
  return false;
}

}  // namespace spf
