// bwd_tma.cuh -- backward of the SP region, rows streamed through shared
// memory by the Tensor Memory Accelerator (bulk copies + mbarriers).
//
// One persistent CTA per SM owns a contiguous block of token rows.  A
// producer warp keeps a ring of nst stages full; a stage holds rb
// consecutive rows and is filled with one bulk copy per input tensor (dy, h,
// dh_out, mask) on the stage's "full" mbarrier.  Rows go to the nrg row
// groups round robin (row i to group i % nrg); a row group (tpr threads)
// computes its row from shared memory and releases the row's stage on its
// "empty" mbarrier.  The loads of up to nst*rb rows are in flight at all
// times, without holding them in registers, so the HBM pipe stays busy
// through the row reductions and the stores.  With the 512-thread block dy
// and xhat stay in registers between the two passes over a row; the
// 544-thread block (two 8-warp row groups, fewer registers) reads them from
// shared memory again.  gamma sits in shared memory as fp32.
// dgamma/dbeta accumulate in registers per thread-owned column; at the end
// the row groups' sums go to the idle ring, are added in row-group order and
// written as one fp32 partial row per CTA, which sp_colsum_kernel reduces in
// CTA order.
//
// If a wait times out (a copy that never lands), the CTA stops, waits (with a
// limit) for what it issued, poisons its dgamma/dbeta partial with NaN so the
// failure is visible in the result, and reports it in the device status word.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace spf {

constexpr int kBwdTmaNarrowBlock = 512;  // the 16-warp block (128 registers)
constexpr int kBwdTmaMidBlock = 544;     // two 8-warp row groups + producer (96 registers)


// NTHR = 512: at most 16 warps (15 consumer + 1 producer), so 128 registers
// per thread fit every SM sub-partition's register file; the 544-thread
// block trades registers for warps (96 registers).  KEEP: dy and xhat stay
// in registers between the two passes (VPT <= 3, 512 threads); otherwise
// pass 2 reads them from shared memory again.  MASK: the keep bits come
// from the stored mask; REGEN: they are recomputed from the seed (no mask
// stored), before the row's data is waited for.
template <bool LN, int VPT, bool DH, bool MASK, bool REGEN, int NTHR>
__global__ void __launch_bounds__(NTHR, 1) sp_bwd_tma_kernel(const BwdArgs a, const BwdTmaLayout L) {
  constexpr bool KEEP = VPT <= 3 && NTHR <= 512;
  constexpr int EV = 8;
  constexpr int NS = LN ? 2 : 1;
  __shared__ float red[2 * 32 * 2];
  __shared__ int s_failed;  // set when any wait timed out
  extern __shared__ __align__(16) unsigned char dsm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm);
  uint64_t* empty = full + L.nst;
  // gamma, fp32.  With KEEP as two planes of float4 -- elements 0..3 of
  // every vector, then elements 4..7 -- so a warp's float4 reads for
  // consecutive vectors hit distinct banks.  In the 544-thread block vector
  // by vector with the two float4 halves of vector v swapped when bit 2 of v
  // is set, which also covers all 32 banks per quarter warp with simpler
  // addressing.  Otherwise plain vector by vector: the 4-vector 512-thread
  // backward measured 0.4% slower with the swizzle despite its two-way
  // conflicts.
  constexpr bool kPlanar = KEEP;
  constexpr int kSwz = (!KEEP && NTHR == kBwdTmaMidBlock) ? 1 : 0;
  float* sgam = reinterpret_cast<float*>(dsm + 16 * ((2 * L.nst * 8 + 15) / 16));
  unsigned char* stages = dsm + L.smem_stages;

  // kernel parameters used in the hot loop, held in registers
  const int H = a.H, nvec = a.nvec, tpr = a.tpr, nrg = L.nrg, nst = L.nst, rb = L.rb;
  const float invH = 1.0f / a.Hf;
  const float scale = a.scale;
  const int nthr_cons = nrg * tpr;
  const bool producer = threadIdx.x >= nthr_cons;
  const int rg = producer ? nrg : (int)threadIdx.x / tpr;
  const int lr = (int)threadIdx.x - rg * tpr;
  const int64_t r0 = (int64_t)blockIdx.x * a.rows_per_cta;
  const int64_t r1 = min(a.rows, r0 + a.rows_per_cta);
  const int n = r1 > r0 ? (int)(r1 - r0) : 0;
  const int nstage = (n + rb - 1) / rb;  // stages this CTA fills
  const int nslot = nstage * rb;         // row slots, the last stage padded to rb rows
  const size_t rowb = (size_t)H * 2;

  // Producer: fill stage j (rows j*rb ..) of the ring.
  auto issue_stage = [&](int j, uint64_t pol) {
    if (j == a.drop_stage && blockIdx.x == 0) return;  // test hook: this stage never lands
    const int s = j % nst;
    unsigned char* st = stages + (size_t)s * L.stage_bytes;
    const int64_t r = r0 + (int64_t)j * rb;
    const int rows = min(rb, n - j * rb);
    const uint32_t bb = (uint32_t)(rows * rowb);  // bytes of one bf16 tensor's rows
    mbar_arrive_expect_tx(&full[s], bb * (DH ? 3u : 2u) + (MASK ? (uint32_t)(rows * H) : 0u));
    tma_load_1d(st, reinterpret_cast<const char*>(a.dy) + r * rowb, bb, &full[s], pol);
    tma_load_1d(st + L.off_h, reinterpret_cast<const char*>(a.h) + r * rowb, bb, &full[s], pol);
    if constexpr (DH)
      tma_load_1d(st + L.off_dh, reinterpret_cast<const char*>(a.dh) + r * rowb, bb, &full[s], pol);
    if constexpr (MASK)
      tma_load_1d(st + L.off_mask, a.mask + r * (int64_t)H, (uint32_t)(rows * H), &full[s], pol);
  };
  const bool lead = producer && lr == 0;
  int issued = 0;
  if (lead && n > 0 && n <= nst * rb) {
    // the CTA's rows all fit the first ring: the first pf_stages stages head
    // for L2 while the previous kernel drains, so the first rows land early
    // (with more rows per CTA the start-up is a small share of the kernel
    // and early requests only compete with it).  Prefetching every stage
    // instead measured slower: the requests of all stages then arrive
    // together and the first rows wait for the last.
    for (int j = 0; j < min(nstage, L.pf_stages); ++j) {
      const int64_t r = r0 + (int64_t)j * rb;
      const int rows = min(rb, n - j * rb);
      const uint32_t pb = (uint32_t)(rows * rowb);
      l2_prefetch(reinterpret_cast<const char*>(a.dy) + r * rowb, pb);
      l2_prefetch(reinterpret_cast<const char*>(a.h) + r * rowb, pb);
      if constexpr (DH) l2_prefetch(reinterpret_cast<const char*>(a.dh) + r * rowb, pb);
      if constexpr (MASK) l2_prefetch(a.mask + r * (int64_t)H, (uint32_t)(rows * H));
    }
  }
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (lead) {
    s_failed = 0;
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], (uint32_t)(rb * tpr));  // the stage's row groups release
    }
    fence_mbar_init();
    // the first ring's worth of rows goes out before anything else happens
    const uint64_t pol = policy_evict_first();
    for (; issued < min(nstage, nst); ++issued) issue_stage(issued, pol);
  } else if (!producer) {
    for (int i = threadIdx.x; i < nvec; i += nthr_cons) {
      float g[EV];
      Act16<__nv_bfloat16>::unpack(ld_cached(reinterpret_cast<const __nv_bfloat16*>(a.gamma) + i * EV), g);
      const int sw = (i >> 2) & kSwz;
      reinterpret_cast<float4*>(sgam)[kPlanar ? i : 2 * i + sw] = make_float4(g[0], g[1], g[2], g[3]);
      reinterpret_cast<float4*>(sgam)[kPlanar ? nvec + i : 2 * i + (sw ^ 1)] =
          make_float4(g[4], g[5], g[6], g[7]);
    }
  }
  __syncthreads();

  bool ok = true;
  f2_t dg[VPT][4];
  f2_t db[LN ? VPT : 1][4];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dg[k][q] = f2(0.f, 0.f);
      if constexpr (LN) db[k][q] = f2(0.f, 0.f);
    }
  }

  if (producer) {
    if (lead) {
      const uint64_t pol = policy_evict_first();
      for (int j = issued; j < nstage; ++j) {
        const int k = j / nst;  // >= 1: the slot was used k times before
        if (!mbar_wait(&empty[j % nst], (uint32_t)((k - 1) & 1), a.wait_ns)) {
          ok = false;
          break;
        }
        issue_stage(j, pol);
        issued = j + 1;
      }
      // nothing may still be landing in shared memory when the ring is
      // reused below or the CTA exits; a copy that did not land in time
      // leaves the ring unusable
      for (int j = max(0, issued - nst); j < issued; ++j)
        if (!mbar_wait(&full[j % nst], (uint32_t)((j / nst) & 1), a.wait_ns)) ok = false;
    }
  } else {
    float* rred = red + rg * 2 * (tpr >> 5) * NS;
    int slot = 0;
    // the last vector slot of a thread may fall beyond the row
    const bool last_in = lr + (VPT - 1) * tpr < nvec;
    // row statistics one row ahead, so their DRAM latency hides behind a row
    float rstd_n = 0.f, mu_n = 0.f;
    if (rg < n) {
      rstd_n = __ldcs(a.rstd + r0 + rg);
      if constexpr (LN) mu_n = __ldcs(a.mean + r0 + rg);
    }
    const f2_t sc = f2(scale, scale);
    // row slot i, its stage j = i / rb, the stage's row ri = i % rb, ring
    // slot s = j % nst and phase parity (j / nst) & 1.  In the 512-thread
    // block rb divides nrg, so iteration jj is stage jj * (nrg / rb) + rg / rb
    // and ri = rg % rb throughout, which keeps its register budget; the
    // 544-thread block keeps them incrementally.
    constexpr bool kStageMajor = NTHR <= kBwdTmaNarrowBlock;
    int ri = rg % rb, s = (rg / rb) % nst, par = ((rg / rb) / nst) & 1;
    for (int i = rg, jj = 0; i < nslot; i += nrg, ++jj) {
      if constexpr (kStageMajor) {
        const int j = jj * (nrg / rb) + rg / rb;
        s = j % nst;
        par = (j / nst) & 1;
      } else if (i != rg) {
        ri += nrg;
        while (ri >= rb) {
          ri -= rb;
          if (++s == nst) {
            s = 0;
            par ^= 1;
          }
        }
      }
      uint32_t keep[REGEN ? VPT : 1];
      if constexpr (REGEN) {  // depends only on the element index: before the wait
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int v = lr + k * tpr;
          keep[k] = 0xFFu;
          if (i < n && (k < VPT - 1 || last_in)) {
            const uint64_t g0 = (uint64_t)((a.grow0 + r0 + i) * (int64_t)H + (int64_t)v * EV);
            keep[k] = keep_bits4(g0 >> 2, a.keys, a.thr) | (keep_bits4((g0 >> 2) + 1, a.keys, a.thr) << 4);
          }
        }
      }
      // the whole row group agrees on the outcome of the wait before any of
      // it enters the row reduction's named barrier
      // (one-warp row groups vote; wider ones use their named barrier, id <= 8)
      const bool landed = mbar_wait(&full[s], (uint32_t)par, a.wait_ns);
      const bool all_landed =
          tpr == 32 ? __all_sync(0xFFFFFFFFu, landed) : bar_red_and(1 + rg, tpr, landed);
      if (!all_landed) {
        ok = false;
        break;
      }
      if (i >= n) {  // padding of the last stage: just release it
        mbar_arrive(&empty[s]);
        continue;
      }
      const unsigned char* st = stages + (size_t)s * L.stage_bytes;
      const int64_t r = r0 + i;
      const size_t rofs = (size_t)ri * rowb;  // this row inside each tensor's block
      const uint4* sdy = reinterpret_cast<const uint4*>(st + rofs);
      const uint4* sh = reinterpret_cast<const uint4*>(st + L.off_h + rofs);
      const uint4* sdh = reinterpret_cast<const uint4*>(st + L.off_dh + rofs);
      const uint8_t* smk = st + L.off_mask + (size_t)ri * H;
      const float rstd = rstd_n;
      const float mu = mu_n;
      if (i + nrg < n) {
        rstd_n = __ldcs(a.rstd + r + nrg);
        if constexpr (LN) mu_n = __ldcs(a.mean + r + nrg);
      }
      const f2_t r2 = f2(rstd, rstd), mu2 = f2(mu, mu);

      // pass 1: xhat = (h-mu)*rstd and g = gamma*dy; row sums of g*xhat (and
      // g); the dgamma/dbeta contributions dy*xhat (and dy).  With KEEP, g and
      // xhat stay in registers for pass 2.
      f2_t gk[KEEP ? VPT : 1][4], xhk[KEEP ? VPT : 1][4];
      f2_t sgx = f2(0.f, 0.f), sg = f2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lr + k * tpr;
        if (k < VPT - 1 || last_in) {
          const uint4 wdy = sdy[v], wh = sh[v];
          const float4* gp = kPlanar ? reinterpret_cast<const float4*>(sgam) + v
                                     : reinterpret_cast<const float4*>(sgam + v * EV);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 g4 = kPlanar ? gp[(q >> 1) * nvec] : gp[(q >> 1) ^ ((v >> 2) & kSwz)];
            const f2_t gm = (q & 1) ? f2(g4.z, g4.w) : f2(g4.x, g4.y);
            const f2_t dy = bf2_to_f2(reinterpret_cast<const uint32_t*>(&wdy)[q]);
            const f2_t hq = bf2_to_f2(reinterpret_cast<const uint32_t*>(&wh)[q]);
            const f2_t xh = (KEEP && !LN) ? f2_mul(hq, r2) : f2_mul(f2_sub(hq, mu2), r2);  // RMS: mean 0
            const f2_t g = f2_mul(gm, dy);
            if constexpr (KEEP) {
              gk[k][q] = g;
              xhk[k][q] = xh;
              dg[k][q] = f2_fma(dy, xh, dg[k][q]);
              if constexpr (LN) db[k][q] = f2_add(db[k][q], dy);
            }
            sgx = f2_fma(g, xh, sgx);
            if constexpr (LN) sg = f2_add(sg, g);
          }
        }
      }
      float sums[NS];
      {
        float lo, hi;
        f2_split(sgx, lo, hi);
        sums[0] = lo + hi;
        if constexpr (LN) {
          f2_split(sg, lo, hi);
          sums[NS - 1] = lo + hi;
        }
      }
      row_allreduce<NS>(sums, tpr, lr, 1 + rg, rred, slot);
      slot ^= 1;
      const f2_t ncgx = f2(-sums[0] * invH, -sums[0] * invH);
      const float cgs = LN ? sums[NS - 1] * invH : 0.f;
      const f2_t cg = f2(cgs, cgs);

      // pass 2: dH, d_residual, d_sum (without KEEP also the dgamma/dbeta
      // contributions, from dy and h read again)
      __nv_bfloat16* dres_row = reinterpret_cast<__nv_bfloat16*>(a.d_res) + r * (int64_t)H;
      __nv_bfloat16* dsum_row = reinterpret_cast<__nv_bfloat16*>(a.d_sum) + r * (int64_t)H;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lr + k * tpr;
        if (k < VPT - 1 || last_in) {
          const float4* gp = reinterpret_cast<const float4*>(sgam + v * EV);  // !KEEP only
          uint4 wdh = make_uint4(0u, 0u, 0u, 0u);
          if constexpr (DH) wdh = sdh[v];
          // the stored mask is applied to the packed bf16 output as byte
          // masks; the regenerated mask uses keep bits
          constexpr bool kByteMask = MASK && NTHR <= kBwdTmaMidBlock;
          uint32_t mk = 0xFFu;
          uint2 mbytes = make_uint2(0u, 0u);  // each mask byte as 0x00 / 0xFF
          if constexpr (kByteMask) {
            mbytes = *reinterpret_cast<const uint2*>(smk + v * EV);
            mbytes.x = (mbytes.x & 0x01010101u) * 0xFFu;
            mbytes.y = (mbytes.y & 0x01010101u) * 0xFFu;
          } else if constexpr (MASK) {
            mk = ld_mask_shared8(smk + v * EV);
          }
          if constexpr (REGEN) mk = keep[k];
          uint4 wdy2 = make_uint4(0u, 0u, 0u, 0u), wh2 = make_uint4(0u, 0u, 0u, 0u);
          if constexpr (!KEEP) {
            wdy2 = sdy[v];
            wh2 = sh[v];
          }
          uint32_t wres[4], wsum[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            f2_t g, xh, dy;
            if constexpr (KEEP) {
              g = gk[k][q];
              xh = xhk[k][q];
            } else {
              const float4 g4 = gp[(q >> 1) ^ ((v >> 2) & kSwz)];
              const f2_t gm = (q & 1) ? f2(g4.z, g4.w) : f2(g4.x, g4.y);
              dy = bf2_to_f2(reinterpret_cast<const uint32_t*>(&wdy2)[q]);
              xh = f2_mul(f2_sub(bf2_to_f2(reinterpret_cast<const uint32_t*>(&wh2)[q]), mu2), r2);
              g = f2_mul(gm, dy);
            }
            // rstd * (g - mean(g) - xhat * mean(g xhat)) + dh_out
            const f2_t t = (KEEP && !LN) ? f2_fma(xh, ncgx, g) : f2_fma(xh, ncgx, f2_sub(g, cg));
            f2_t dres;
            if constexpr (DH)
              dres = f2_fma(r2, t, bf2_to_f2(reinterpret_cast<const uint32_t*>(&wdh)[q]));
            else
              dres = f2_mul(r2, t);
            f2_t dsum = f2_mul(dres, sc);
            if constexpr ((MASK && !kByteMask) || REGEN) {
              float sl, sh2;
              f2_split(dsum, sl, sh2);
              dsum = f2(((mk >> (2 * q)) & 1u) ? sl : 0.f, ((mk >> (2 * q + 1)) & 1u) ? sh2 : 0.f);
            }
            wres[q] = f2_to_bf2(dres);
            wsum[q] = f2_to_bf2(dsum);
            if constexpr (kByteMask) {
              // a dropped element's bf16 becomes +0, as if its product were 0:
              // the 16-bit halves take the 0x00/0xFF bytes of elements 2q, 2q+1
              const uint32_t mb = (q < 2) ? mbytes.x : mbytes.y;
              wsum[q] &= __byte_perm(mb, 0u, (q & 1) ? 0x3322u : 0x1100u);
            }
            if constexpr (!KEEP) {
              dg[k][q] = f2_fma(dy, xh, dg[k][q]);
              if constexpr (LN) db[k][q] = f2_add(db[k][q], dy);
            }
          }
          st_stream(dres_row + v * EV, make_uint4(wres[0], wres[1], wres[2], wres[3]));
          st_stream(dsum_row + v * EV, make_uint4(wsum[0], wsum[1], wsum[2], wsum[3]));
        }
      }
      mbar_arrive(&empty[s]);
    }
  }

  if (!ok) s_failed = 1;
  __syncthreads();  // every stage consumed and landed (unless a wait timed out)
  // A CTA whose wait timed out poisons its partial rows so dgamma/dbeta are
  // NaN, and leaves the ring alone: a copy may still be landing there.
  if (s_failed != 0) {
    if (threadIdx.x == 0) report_status(a.status, kStatusBwdWaitTimeout);
    for (int st = 0; st < NS; ++st)
      for (int c = threadIdx.x; c < H; c += blockDim.x)
        __stcg(a.ws + ((int64_t)st * a.nparts + blockIdx.x) * H + c, __int_as_float(0x7FC00000));
    return;
  }

  // ---- dgamma/dbeta: row groups' column sums into the ring, added in order ---
  // The ring holds them as [nrg][NS][H] fp32: each thread stores the 8
  // columns of each of its vectors as two float4; then each thread adds one
  // float4 of columns over the row groups in group order (all the group
  // loads in flight before the adds) and writes it to the CTA's partial row.
  float* part = reinterpret_cast<float*>(stages);
  if (!producer) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lr + k * tpr;
      if (v < nvec) {
        float e[2][8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f2_split(dg[k][q], e[0][2 * q], e[0][2 * q + 1]);
          if constexpr (LN) f2_split(db[k][q], e[1][2 * q], e[1][2 * q + 1]);
        }
#pragma unroll
        for (int st = 0; st < NS; ++st) {
          float4* dst = reinterpret_cast<float4*>(part + ((size_t)rg * NS + st) * H + (size_t)v * EV);
          dst[0] = make_float4(e[st][0], e[st][1], e[st][2], e[st][3]);
          dst[1] = make_float4(e[st][4], e[st][5], e[st][6], e[st][7]);
        }
      }
    }
  }
  __syncthreads();
  const int n4 = NS * H / 4;  // float4 columns of both statistics
  const size_t gstride4 = (size_t)NS * H / 4;
  for (int c4 = threadIdx.x; c4 < n4; c4 += blockDim.x) {
    const float4* src = reinterpret_cast<const float4*>(part) + c4;
    float4 acc = src[0];
    for (int g0 = 1; g0 < nrg; g0 += 8) {
      float4 t[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (g0 + u < nrg) t[u] = src[(size_t)(g0 + u) * gstride4];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (g0 + u < nrg) {
          acc.x += t[u].x;
          acc.y += t[u].y;
          acc.z += t[u].z;
          acc.w += t[u].w;
        }
      }
    }
    const int st = (c4 * 4) / H, c = c4 * 4 - st * H;
    __stcg(reinterpret_cast<float4*>(a.ws + ((int64_t)st * a.nparts + blockIdx.x) * H + c), acc);
  }
}

}  // namespace spf
