// fwd.cuh -- forward of the SP region: reduce -> dropout -> residual -> norm.
//
// One token row per row group of `tpr` threads (one warp for H <= 1024 bf16,
// several warps for larger H); each thread owns VPT 16-byte vectors of the
// row, strided by tpr so every warp access is 512 contiguous bytes.  All
// T partial vectors, the residual and gamma/beta of a thread are requested
// before any of them is used, so each thread keeps (T+2)*VPT*16 bytes in
// flight.  The rounded residual stream stays in registers for the norm: HBM
// is read once per input and written once per output.
#pragma once

#include "common.cuh"

namespace spf {

template <typename Act, int T, bool LN, int VPT>
__global__ void __launch_bounds__(512) sp_fwd_kernel(const FwdArgs a) {
  using V = Act16<Act>;
  constexpr int EV = V::EV;
  __shared__ float red[2 * 32 * 2];

  const int tpr = a.tpr;
  const int rg = threadIdx.x / tpr;
  const int lr = threadIdx.x - rg * tpr;
  const int rpc = blockDim.x / tpr;
  const int64_t r = (int64_t)blockIdx.x * rpc + rg;

  grid_dep_wait();
  grid_dep_launch_dependents();
  if (r >= a.rows) return;  // whole row groups leave together

  const int64_t grow = a.grow0 + r;
  const Act* __restrict__ res = reinterpret_cast<const Act*>(a.residual) + r * (int64_t)a.H;
  const int64_t poff = grow * (int64_t)a.H;

  // ---- issue every load of the row before using any of them --------------
  uint4 pv[VPT][T];
  uint4 rv[VPT];
  uint4 gv[VPT];
  uint4 bv[LN ? VPT : 1];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lr + k * tpr;
    if (v < a.nvec) {
#pragma unroll
      for (int t = 0; t < T; ++t)
        pv[k][t] = ld_stream(reinterpret_cast<const Act*>(a.P[t]) + poff + (int64_t)v * EV);
      rv[k] = ld_stream(res + (int64_t)v * EV);
      gv[k] = ld_cached(reinterpret_cast<const Act*>(a.gamma) + v * EV);
      if constexpr (LN) bv[k] = ld_cached(reinterpret_cast<const Act*>(a.beta) + v * EV);
    }
  }

  // ---- reduce, mask, dropout, residual add; store h and the mask ---------
  float hr[VPT][EV];
  float s = 0.f;  // row sum (LN) or sum of squares (RMS) of the stored h
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lr + k * tpr;
#pragma unroll
    for (int e = 0; e < EV; ++e) hr[k][e] = 0.f;
    if (v < a.nvec) {
      float acc[EV], tmp[EV], rs[EV];
      V::unpack(pv[k][0], acc);
#pragma unroll
      for (int t = 1; t < T; ++t) {
        V::unpack(pv[k][t], tmp);
#pragma unroll
        for (int e = 0; e < EV; ++e) acc[e] += tmp[e];
      }
      V::unpack(rv[k], rs);
      const uint64_t g0 = (uint64_t)(poff + (int64_t)v * EV);  // global index of element 0
      uint32_t keep = (1u << EV) - 1u;
      if (a.dropout) {
        keep = keep_bits4(g0 >> 2, a.key0, a.key1, a.thr);
        if constexpr (EV == 8) keep |= keep_bits4((g0 >> 2) + 1, a.key0, a.key1, a.thr) << 4;
      }
      uint4 hp;
      if constexpr (EV == 8) {
        uint32_t hb[EV];
#pragma unroll
        for (int e = 0; e < EV; ++e)
          hb[e] = residual_bf16(rs[e], acc[e], a.scale, a.scale_lo, (keep >> e) & 1u);
        hp = make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16),
                        hb[6] | (hb[7] << 16));
      } else {
        float hv[EV];
#pragma unroll
        for (int e = 0; e < EV; ++e) hv[e] = rs[e] + (((keep >> e) & 1u) ? acc[e] * a.scale : 0.f);
        hp = V::pack(hv);
      }
      st_stream(reinterpret_cast<Act*>(a.h) + r * (int64_t)a.H + (int64_t)v * EV, hp);
      if (a.mask) st_mask<EV>(a.mask + r * (int64_t)a.H + (int64_t)v * EV, keep);
      V::unpack(hp, hr[k]);  // the norm reads the stored (rounded) value
#pragma unroll
      for (int e = 0; e < EV; ++e) s += LN ? hr[k][e] : hr[k][e] * hr[k][e];
    }
  }

  // ---- row statistics ------------------------------------------------------
  float* rred = red + rg * 2 * (tpr >> 5);
  float sv[1] = {s};
  row_allreduce<1>(sv, tpr, lr, 1 + rg, rred, 0);
  float mu = 0.f, rstd;
  if constexpr (LN) {
    mu = sv[0] / a.Hf;
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (lr + k * tpr < a.nvec) {
#pragma unroll
        for (int e = 0; e < EV; ++e) {
          const float d = hr[k][e] - mu;
          q += d * d;
        }
      }
    }
    float qv[1] = {q};
    row_allreduce<1>(qv, tpr, lr, 1 + rg, rred, 1);
    rstd = 1.0f / sqrtf(qv[0] / a.Hf + a.eps);
  } else {
    rstd = 1.0f / sqrtf(sv[0] / a.Hf + a.eps);
  }

  // ---- y = gamma * xhat (+ beta), one rounding -----------------------------
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lr + k * tpr;
    if (v < a.nvec) {
      float gm[EV], yv[EV];
      V::unpack(gv[k], gm);
      if constexpr (LN) {
        float bt[EV];
        V::unpack(bv[k], bt);
#pragma unroll
        for (int e = 0; e < EV; ++e) yv[e] = gm[e] * ((hr[k][e] - mu) * rstd) + bt[e];
      } else {
#pragma unroll
        for (int e = 0; e < EV; ++e) yv[e] = gm[e] * (hr[k][e] * rstd);
      }
      st_stream(reinterpret_cast<Act*>(a.y) + r * (int64_t)a.H + (int64_t)v * EV, V::pack(yv));
    }
  }
  if (lr == 0) {
    a.rstd[r] = rstd;
    if constexpr (LN) a.mean[r] = mu;
  }
}

}  // namespace spf
