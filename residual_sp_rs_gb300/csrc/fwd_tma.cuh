// fwd_tma.cuh -- forward of the SP region with rows streamed through shared
// memory by the Tensor Memory Accelerator (bf16).
//
// One persistent CTA per SM owns a contiguous block of token rows.  A
// producer warp keeps a ring of nst stages full; a stage holds rb
// consecutive rows of each of the T partials and of the residual, each
// filled with one bulk copy on the stage's "full" mbarrier.  Rows go to the
// nrg consumer row groups round robin (row i to group i % nrg); a group
// reduces, masks, adds and normalises its row from shared memory and
// releases the row's stage on its "empty" mbarrier, so the arithmetic of
// one row overlaps the loads of the next ones.  Small stages (down to one
// row) let the first rows start as soon as they land.  gamma/beta are kept
// in shared memory as fp32.  NTHR is the block size the registers are
// budgeted for: 544 (16 consumer warps + producer, up to 96 registers) or
// 896 (27 + producer, 72 registers) for the many short rows of small T.
//
// The mask depends only on the element index, so a thread draws (and
// stores) its row's keep bits before it waits for the row's data: the
// Philox arithmetic overlaps the loads.
//
// CH (chunked): when a stage of one whole row does not fit twice in shared
// memory (T*H large), a stage holds one column chunk of one row instead --
// the tpr vectors of one vector slot k of every thread (tpr*16 bytes of each
// input) -- so a row is VPT stages, each released as soon as its slot's h is
// in registers.
//
// If a wait times out, the row group stops, writes NaN into the rstd of the
// rows it did not finish and reports the timeout in the device status word.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace spf {

// bf16 residual stream for a pair when 1/(1-p) is not a dyadic fraction
// (s_lo != 0): as residual_bf2, without the tie-to-even branch.  Then the
// exact value E = res + acc*s is not a bf16 midpoint unless acc = 0, and for
// acc = 0, E = res is a bf16 value whose midpoint test (d < 0) needs no tie
// rule.  (p = 0.5, 0.75, ... make s dyadic; those take residual_bf2.)
__device__ __forceinline__ uint32_t residual_bf2_drop(f2_t res, f2_t acc, f2_t s_hi, f2_t s_lo) {
  const f2_t h1 = f2_fma(acc, s_hi, res);
  float h1l, h1h;
  f2_split(h1, h1l, h1h);
  const uint32_t ul = __float_as_uint(h1l), uh = __float_as_uint(h1h);
  const f2_t m = f2(__uint_as_float((ul & 0xFFFF0000u) | 0x8000u),
                    __uint_as_float((uh & 0xFFFF0000u) | 0x8000u));
  const f2_t d = f2_fma(acc, s_lo, f2_fma(acc, s_hi, f2_sub(res, m)));
  const f2_t gap = f2_mul(h1, f2(0x1p12f, 0x1p12f));
  float dl, dh, gl, gh, rl, rh;
  f2_split(d, dl, dh);
  f2_split(gap, gl, gh);
  f2_split(res, rl, rh);
  // past the midpoint, away from zero: d and h1 agree in sign, d != 0
  const uint32_t pl = (int)(__float_as_uint(dl) ^ (ul & 0x80000000u)) > 0 ? 0x1u : 0u;
  const uint32_t ph = (int)(__float_as_uint(dh) ^ (uh & 0x80000000u)) > 0 ? 0x10000u : 0u;
  uint32_t w = __byte_perm(ul, uh, 0x7632) + pl + ph;
  if (fabsf(gl) < fabsf(rl) || fabsf(gh) < fabsf(rh)) {  // rare: |h| < 2^-12 |res|
    float al, ah, shl, shh, sll, slh;
    f2_split(acc, al, ah);
    f2_split(s_hi, shl, shh);
    f2_split(s_lo, sll, slh);
    uint32_t bl = w & 0xFFFFu, bh = w >> 16;
    if (fabsf(gl) < fabsf(rl)) bl = residual_bf16_dd(rl, al, shl, sll, true);
    if (fabsf(gh) < fabsf(rh)) bh = residual_bf16_dd(rh, ah, shh, slh, true);
    w = bl | (bh << 16);
  }
  return w;
}

// The same rounding for one 16-byte vector (four pairs) with a single guard
// branch for the vector instead of one per pair.
__device__ __forceinline__ void residual_vec8_drop(const f2_t (&acc)[4], const f2_t (&res)[4], f2_t s_hi,
                                                   f2_t s_lo, uint32_t (&hw)[4]) {
  bool risky = false;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const f2_t h1 = f2_fma(acc[q], s_hi, res[q]);
    float h1l, h1h;
    f2_split(h1, h1l, h1h);
    const uint32_t ul = __float_as_uint(h1l), uh = __float_as_uint(h1h);
    const f2_t m = f2(__uint_as_float((ul & 0xFFFF0000u) | 0x8000u),
                      __uint_as_float((uh & 0xFFFF0000u) | 0x8000u));
    const f2_t d = f2_fma(acc[q], s_lo, f2_fma(acc[q], s_hi, f2_sub(res[q], m)));
    const f2_t gap = f2_mul(h1, f2(0x1p12f, 0x1p12f));
    float dl, dh, gl, gh, rl, rh;
    f2_split(d, dl, dh);
    f2_split(gap, gl, gh);
    f2_split(res[q], rl, rh);
    const uint32_t pl = (int)(__float_as_uint(dl) ^ (ul & 0x80000000u)) > 0 ? 0x1u : 0u;
    const uint32_t ph = (int)(__float_as_uint(dh) ^ (uh & 0x80000000u)) > 0 ? 0x10000u : 0u;
    hw[q] = __byte_perm(ul, uh, 0x7632) + pl + ph;
    risky |= (fabsf(gl) < fabsf(rl)) | (fabsf(gh) < fabsf(rh));
  }
  if (risky) {  // rare: |h| < 2^-12 |res| somewhere in the vector
    float shl, shh, sll, slh;
    f2_split(s_hi, shl, shh);
    f2_split(s_lo, sll, slh);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float al, ah, rl, rh;
      f2_split(acc[q], al, ah);
      f2_split(res[q], rl, rh);
      uint32_t bl = hw[q] & 0xFFFFu, bh = hw[q] >> 16;
      if (fabsf(__fmaf_rn(al, shl, rl)) * 0x1p12f < fabsf(rl)) bl = residual_bf16_dd(rl, al, shl, sll, true);
      if (fabsf(__fmaf_rn(ah, shh, rh)) * 0x1p12f < fabsf(rh)) bh = residual_bf16_dd(rh, ah, shh, slh, true);
      hw[q] = bl | (bh << 16);
    }
  }
}

// A thread's share of the stored h of its row, as fp32 pairs, for the norm's
// two passes.
template <int VPT>
struct HRow {
  f2_t v[VPT][4];
  __device__ __forceinline__ void set(int k, int q, f2_t f) { v[k][q] = f; }
  __device__ __forceinline__ f2_t get(int k, int q) const { return v[k][q]; }
};

// FAST: p > 0 with 1/(1-p) not dyadic (the common case) -- no tie rule, no
// runtime mode branches in the element loop.  Otherwise GENERIC.

template <int T, bool LN, int VPT, bool FAST, int NTHR, bool CH>
__global__ void __launch_bounds__(NTHR, 1) sp_fwd_tma_kernel(const FwdArgs a, const FwdTmaLayout L) {
  constexpr int EV = 8;
  constexpr int NCH = CH ? VPT : 1;  // stages per row stage (CH: rb == 1)
  __shared__ float red[2 * 32 * 2];
  extern __shared__ __align__(16) unsigned char dsm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm);
  uint64_t* empty = full + L.nst;
  // gamma then beta, fp32, each as two planes of float4 -- elements 0..3 of
  // every vector, then elements 4..7 -- so a warp's reads of consecutive
  // vectors are contiguous (no bank conflicts)
  float* sgb = reinterpret_cast<float*>(dsm + 16 * ((2 * L.nst * 8 + 15) / 16));
  unsigned char* stages = dsm + L.smem_stages;

  const int H = a.H, nvec = a.nvec, tpr = a.tpr;
  const float invH = 1.0f / a.Hf;
  const int nthr_cons = L.nrg * tpr;
  const bool producer = (int)threadIdx.x >= nthr_cons;
  const int rg = producer ? L.nrg : (int)threadIdx.x / tpr;
  const int lr = (int)threadIdx.x - rg * tpr;
  const int64_t r0 = (int64_t)blockIdx.x * L.rows_per_cta;
  const int64_t r1 = min(a.rows, r0 + L.rows_per_cta);
  const int n = r1 > r0 ? (int)(r1 - r0) : 0;
  const int nrow_st = (n + L.rb - 1) / L.rb;  // stages of rb rows (CH: rows)
  const int nstage = nrow_st * NCH;
  const int nslot = nrow_st * L.rb;  // row slots, the last stage padded to rb rows
  const size_t rowb = (size_t)H * 2;
  // the partials and the residual are read once, but an evict-normal policy
  // on their copies measured faster than evict-first at T = 8 (GPT LayerNorm
  // forward 62.1 -> 60.6 us, large-hidden 452 -> 440 us back to back) and
  // the same at the pages' shape
  const uint64_t pol = policy_evict_normal();

  auto issue_stage = [&](int j) {
    if (j == a.drop_stage && blockIdx.x == 0) return;  // test hook: this stage never lands
    const int s = j % L.nst;
    unsigned char* st = stages + (size_t)s * L.stage_bytes;
    const int jr = j / NCH, k = j - jr * NCH;   // row stage and (CH) column chunk
    const int64_t r = r0 + (int64_t)jr * L.rb;  // local row of the stage's first row
    size_t off = 0;
    uint32_t bb;
    if constexpr (CH) {
      off = (size_t)k * L.blk;
      bb = (uint32_t)min((size_t)L.blk, rowb - off);
    } else {
      bb = (uint32_t)(min(L.rb, n - jr * L.rb) * rowb);
    }
    mbar_arrive_expect_tx(&full[s], bb * (uint32_t)(T + 1));
#pragma unroll
    for (int t = 0; t < T; ++t)
      tma_load_1d(st + (size_t)t * L.blk,
                  reinterpret_cast<const char*>(a.P[t]) + (a.grow0 + r) * rowb + off, bb, &full[s], pol);
    tma_load_1d(st + (size_t)T * L.blk, reinterpret_cast<const char*>(a.residual) + r * rowb + off, bb,
                &full[s], pol);
  };

  const bool dropout = a.dropout != 0, nontie = a.dropout && !a.dyadic_scale;
  const bool last_in = lr + (VPT - 1) * tpr < nvec;  // the last vector slot may fall outside
  // The mask depends only on the element index: draw (and store) row slot
  // i's keep bits, before waiting for the row's data.
  auto draw_row = [&](int i, uint32_t (&keep)[VPT]) {
    const int64_t r = r0 + i;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      keep[k] = 0xFFu;
      const int v = lr + k * tpr;
      if ((FAST || dropout) && i < n && (k < VPT - 1 || last_in)) {
        const uint64_t g0 = (uint64_t)((a.grow0 + r) * H + (int64_t)v * EV);
        keep[k] = keep_bits4(g0 >> 2, a.keys, a.thr) | (keep_bits4((g0 >> 2) + 1, a.keys, a.thr) << 4);
        if (a.mask) st_mask<EV>(a.mask + r * (int64_t)H + v * EV, keep[k]);
      }
    }
  };

  const bool lead = producer && lr == 0;
  int issued = 0;
  uint32_t keep[VPT];  // keep bits of this thread's next row, drawn ahead
  if (!CH && lead && n > 0 && n <= L.nst * L.rb) {
    // the CTA's rows all fit the first ring: the first pf_stages stages head
    // for L2 while the previous kernel drains, so the first rows land early
    // (with more rows per CTA the start-up is a small share of the kernel
    // and early requests only compete with it).  Prefetching every stage
    // instead measured slower: the requests of all stages then arrive
    // together and the first rows wait for the last.
    for (int jr = 0; jr < min(nrow_st, L.pf_stages); ++jr) {
      const int64_t r = r0 + (int64_t)jr * L.rb;
      const uint32_t pb = (uint32_t)(min(L.rb, n - jr * L.rb) * rowb);
#pragma unroll
      for (int t = 0; t < T; ++t) l2_prefetch(reinterpret_cast<const char*>(a.P[t]) + (a.grow0 + r) * rowb, pb);
      l2_prefetch(reinterpret_cast<const char*>(a.residual) + r * rowb, pb);
    }
  }
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (lead) {
    for (int s = 0; s < L.nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], (uint32_t)(L.rb * tpr));
    }
    fence_mbar_init();
    for (; issued < min(nstage, L.nst); ++issued) issue_stage(issued);
  } else if (!producer) {
    // gamma/beta loads stay in flight while the first row's mask is drawn
    // (nvec <= VPT * tpr <= VPT * nthr_cons)
    uint4 gw[VPT], bw[LN ? VPT : 1];
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = threadIdx.x + u * nthr_cons;
      if (i < nvec) {
        gw[u] = ld_cached(reinterpret_cast<const __nv_bfloat16*>(a.gamma) + i * EV);
        if constexpr (LN) bw[u] = ld_cached(reinterpret_cast<const __nv_bfloat16*>(a.beta) + i * EV);
      }
    }
    draw_row(rg, keep);
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int i = threadIdx.x + u * nthr_cons;
      if (i < nvec) {
        float g[EV];
        Act16<__nv_bfloat16>::unpack(gw[u], g);
        reinterpret_cast<float4*>(sgb)[i] = make_float4(g[0], g[1], g[2], g[3]);
        reinterpret_cast<float4*>(sgb)[nvec + i] = make_float4(g[4], g[5], g[6], g[7]);
        if constexpr (LN) {
          Act16<__nv_bfloat16>::unpack(bw[u], g);
          reinterpret_cast<float4*>(sgb + H)[i] = make_float4(g[0], g[1], g[2], g[3]);
          reinterpret_cast<float4*>(sgb + H)[nvec + i] = make_float4(g[4], g[5], g[6], g[7]);
        }
      }
    }
  }
  __syncthreads();

  if (producer) {
    if (lead) {
      for (int j = issued; j < nstage; ++j) {
        const int k = j / L.nst;
        if (!mbar_wait(&empty[j % L.nst], (uint32_t)((k - 1) & 1), a.wait_ns)) {
          report_status(a.status, kStatusFwdWaitTimeout);
          break;
        }
        issue_stage(j);
        issued = j + 1;
      }
      // nothing may still be landing in shared memory when the CTA exits
      for (int j = max(0, issued - L.nst); j < issued; ++j)
        mbar_wait(&full[j % L.nst], (uint32_t)((j / L.nst) & 1), a.wait_ns);
    }
    return;
  }

  float* rred = red + rg * 2 * (tpr >> 5);
  const f2_t shi = f2(a.scale, a.scale), slo = f2(a.scale_lo, a.scale_lo);
  // row slot i, its row stage jr = i / rb, the stage's row ri = i % rb, the
  // ring slot s = (jr * NCH) % nst of its first stage and that stage's phase
  // parity ((jr * NCH) / nst) & 1, kept incrementally
  int ri = rg % L.rb, s = ((rg / L.rb) * NCH) % L.nst, par = (((rg / L.rb) * NCH) / L.nst) & 1;
  // wait for ring slot (s, par) -- the whole row group agrees -- or give up
  auto wait_stage = [&](int ws, int wpar, int i) -> bool {
    const bool landed = mbar_wait(&full[ws], (uint32_t)wpar, a.wait_ns);
    const bool all_landed =
        tpr == 32 ? __all_sync(0xFFFFFFFFu, landed) : bar_red_and(1 + rg, tpr, landed);
    if (!all_landed && lr == 0) {  // mark this row group's unfinished rows
      for (int k = i; k < n; k += L.nrg) a.rstd[r0 + k] = __int_as_float(0x7FC00000);
      report_status(a.status, kStatusFwdWaitTimeout);
    }
    return all_landed;
  };
  for (int i = rg; i < nslot; i += L.nrg) {
    if (i != rg) {
      ri += L.nrg;
      while (ri >= L.rb) {
        ri -= L.rb;
#pragma unroll
        for (int c = 0; c < NCH; ++c)
          if (++s == L.nst) {
            s = 0;
            par ^= 1;
          }
      }
    }
    const int64_t r = r0 + i;

    if (!CH && !wait_stage(s, par, i)) return;
    if (i >= n) {  // padding of the last stage (never with CH: rb == 1)
      if constexpr (!CH) mbar_arrive(&empty[s]);
      continue;
    }
    const unsigned char* st = stages + (size_t)s * L.stage_bytes + (size_t)ri * rowb;
    int cs = s, cpar = par;  // CH: the ring slot of column chunk k
    __nv_bfloat16* h_row = reinterpret_cast<__nv_bfloat16*>(a.h) + r * (int64_t)H;
    __nv_bfloat16* y_row = reinterpret_cast<__nv_bfloat16*>(a.y) + r * (int64_t)H;

    // ---- reduce, dropout, residual add; store h ----------------------------
    // h stays in registers for the norm, as fp32 pairs
    HRow<VPT> hf;
    f2_t s2 = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lr + k * tpr;
      // this thread's vector of slot k: vector vi of each tensor block at sb
      const unsigned char* sb = st;
      int vi = v;
      if constexpr (CH) {
        if (k > 0 && ++cs == L.nst) {
          cs = 0;
          cpar ^= 1;
        }
        if (!wait_stage(cs, cpar, i)) return;
        sb = stages + (size_t)cs * L.stage_bytes;
        vi = lr;
      }
      if (k < VPT - 1 || last_in) {
        uint4 pw[T];
#pragma unroll
        for (int t = 0; t < T; ++t) pw[t] = reinterpret_cast<const uint4*>(sb + (size_t)t * L.blk)[vi];
        const uint4 rw = reinterpret_cast<const uint4*>(sb + (size_t)T * L.blk)[vi];
        const uint32_t kb = keep[k];
        uint32_t hw[4];
        if constexpr (FAST) {
          f2_t acc[4], res[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[q] = bf2_to_f2(reinterpret_cast<const uint32_t*>(&pw[0])[q]);
#pragma unroll
            for (int t = 1; t < T; ++t)
              acc[q] = f2_add(acc[q], bf2_to_f2(reinterpret_cast<const uint32_t*>(&pw[t])[q]));
            float al, ah;
            f2_split(acc[q], al, ah);
            acc[q] = f2(((kb >> (2 * q)) & 1u) ? al : 0.f, ((kb >> (2 * q + 1)) & 1u) ? ah : 0.f);
            res[q] = bf2_to_f2(reinterpret_cast<const uint32_t*>(&rw)[q]);
          }
          residual_vec8_drop(acc, res, shi, slo, hw);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const f2_t hq = bf2_to_f2(hw[q]);
            hf.set(k, q, hq);
            s2 = LN ? f2_add(s2, hq) : f2_fma(hq, hq, s2);
          }
        } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f2_t acc = bf2_to_f2(reinterpret_cast<const uint32_t*>(&pw[0])[q]);
#pragma unroll
          for (int t = 1; t < T; ++t)
            acc = f2_add(acc, bf2_to_f2(reinterpret_cast<const uint32_t*>(&pw[t])[q]));
          const f2_t res = bf2_to_f2(reinterpret_cast<const uint32_t*>(&rw)[q]);
          if (dropout) {
            float al, ah;
            f2_split(acc, al, ah);
            acc = f2(((kb >> (2 * q)) & 1u) ? al : 0.f, ((kb >> (2 * q + 1)) & 1u) ? ah : 0.f);
          }
          hw[q] = nontie ? residual_bf2_drop(res, acc, shi, slo) : residual_bf2(res, acc, shi, slo);
          const f2_t hq = bf2_to_f2(hw[q]);
          hf.set(k, q, hq);
          s2 = LN ? f2_add(s2, hq) : f2_fma(hq, hq, s2);
        }
        }
        st_stream(h_row + v * EV, make_uint4(hw[0], hw[1], hw[2], hw[3]));
      }
      if constexpr (CH) mbar_arrive(&empty[cs]);  // this chunk is no longer read
    }
    if constexpr (!CH) mbar_arrive(&empty[s]);  // the stage is no longer read

    // ---- row statistics -----------------------------------------------------
    float sv[1];
    {
      float lo, hi;
      f2_split(s2, lo, hi);
      sv[0] = lo + hi;
    }
    row_allreduce<1>(sv, tpr, lr, 1 + rg, rred, 0);
    float mu = 0.f, rstd;
    if constexpr (LN) {
      mu = sv[0] * invH;
      const f2_t mu2 = f2(mu, mu);
      f2_t q2 = f2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (k < VPT - 1 || last_in) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const f2_t dd = f2_sub(hf.get(k, q), mu2);
            q2 = f2_fma(dd, dd, q2);
          }
        }
      }
      float qv[1];
      {
        float lo, hi;
        f2_split(q2, lo, hi);
        qv[0] = lo + hi;
      }
      row_allreduce<1>(qv, tpr, lr, 1 + rg, rred, 1);
      rstd = 1.0f / sqrtf(qv[0] * invH + a.eps);
    } else {
      rstd = 1.0f / sqrtf(sv[0] * invH + a.eps);
    }

    // ---- y = gamma * xhat (+ beta), one rounding ------------------------------
    const f2_t r2 = f2(rstd, rstd), mu2 = f2(mu, mu);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lr + k * tpr;
      if (k < VPT - 1 || last_in) {
        const float4* gp = reinterpret_cast<const float4*>(sgb) + v;
        uint32_t yw[4];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const float4 g4 = gp[q2 * nvec];
          const f2_t ga = f2(g4.x, g4.y), gb = f2(g4.z, g4.w);
          if constexpr (LN) {
            const float4 b4 = (reinterpret_cast<const float4*>(sgb + H) + v)[q2 * nvec];
            yw[2 * q2] = f2_to_bf2(f2_fma(ga, f2_mul(f2_sub(hf.get(k, 2 * q2), mu2), r2), f2(b4.x, b4.y)));
            yw[2 * q2 + 1] =
                f2_to_bf2(f2_fma(gb, f2_mul(f2_sub(hf.get(k, 2 * q2 + 1), mu2), r2), f2(b4.z, b4.w)));
          } else {
            yw[2 * q2] = f2_to_bf2(f2_mul(ga, f2_mul(hf.get(k, 2 * q2), r2)));
            yw[2 * q2 + 1] = f2_to_bf2(f2_mul(gb, f2_mul(hf.get(k, 2 * q2 + 1), r2)));
          }
        }
        st_keep(y_row + v * EV, make_uint4(yw[0], yw[1], yw[2], yw[3]));
      }
    }
    if (lr == 0) {
      a.rstd[r] = rstd;
      if constexpr (LN) a.mean[r] = mu;
    }
    draw_row(i + L.nrg, keep);  // the next row's mask, before its data is waited for
  }
}

}  // namespace spf
