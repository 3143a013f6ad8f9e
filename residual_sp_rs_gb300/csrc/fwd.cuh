// fwd.cuh -- forward of the SP region: reduce -> dropout -> residual -> norm.
//
// One token row per row group of `tpr` threads (one warp for H <= 1024 bf16,
// several warps for larger H); each thread owns VPT 16-byte vectors of the
// row, strided by tpr so every warp access is 512 contiguous bytes.  All
// T partial vectors and the residual of a thread are requested before any of
// them is used, so each thread keeps (T+1)*VPT*16 bytes in flight; gamma and
// beta are staged once per CTA in shared memory meanwhile.  The stored
// (rounded) residual stream stays in registers, packed, for the norm: HBM is
// read once per input and written once per output.
#pragma once

#include "common.cuh"

namespace spf {

template <typename Act, int T, bool LN, int VPT>
__global__ void __launch_bounds__(512) sp_fwd_kernel(const FwdArgs a) {
  using V = Act16<Act>;
  constexpr int EV = V::EV;
  __shared__ float red[2 * 32 * 2];
  extern __shared__ uint4 sgb[];  // gamma vectors [nvec] (then beta [nvec] for LN)

  const int tpr = a.tpr;
  const int rg = threadIdx.x / tpr;
  const int lr = threadIdx.x - rg * tpr;
  const int rpc = blockDim.x / tpr;
  const int64_t r = (int64_t)blockIdx.x * rpc + rg;
  const bool active = r < a.rows;  // whole row groups are active or not

  grid_dep_wait();
  grid_dep_launch_dependents();

  const int64_t grow = a.grow0 + r;
  const Act* __restrict__ res = reinterpret_cast<const Act*>(a.residual) + r * (int64_t)a.H;
  const int64_t poff = grow * (int64_t)a.H;

  // ---- issue every load of the row before using any of them --------------
  uint4 pv[VPT][T];
  uint4 rv[VPT];
  if (active) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lr + k * tpr;
      if (v < a.nvec) {
#pragma unroll
        for (int t = 0; t < T; ++t)
          pv[k][t] = ld_stream(reinterpret_cast<const Act*>(a.P[t]) + poff + (int64_t)v * EV);
        rv[k] = ld_stream(res + (int64_t)v * EV);
      }
    }
  }
  // gamma (and beta) once per CTA into shared memory while the row loads fly
  for (int i = threadIdx.x; i < a.nvec; i += blockDim.x) {
    sgb[i] = ld_cached(reinterpret_cast<const Act*>(a.gamma) + i * EV);
    if constexpr (LN) sgb[a.nvec + i] = ld_cached(reinterpret_cast<const Act*>(a.beta) + i * EV);
  }
  __syncthreads();
  if (!active) return;

  // ---- reduce, mask, dropout, residual add; store h and the mask ---------
  // bf16: everything in packed fp32 pairs; hf keeps the stored h for the norm.
  // f32: plain fp32 lanes; hp keeps the stored h.
  f2_t hf[EV == 8 ? VPT : 1][4];
  uint4 hp[EV == 8 ? 1 : VPT];
  f2_t s2 = f2(0.f, 0.f);  // row sum (LN) or sum of squares (RMS), as pairs
  float s = 0.f;           // the same for f32
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lr + k * tpr;
    if (v < a.nvec) {
      const uint64_t g0 = (uint64_t)(poff + (int64_t)v * EV);  // global index of element 0
      uint32_t keep = (1u << EV) - 1u;
      if (a.dropout) {
        keep = keep_bits4(g0 >> 2, a.keys, a.thr);
        if constexpr (EV == 8) keep |= keep_bits4((g0 >> 2) + 1, a.keys, a.thr) << 4;
      }
      uint4 hout;
      if constexpr (EV == 8) {
        const f2_t shi = f2(a.scale, a.scale), slo = f2(a.scale_lo, a.scale_lo);
        uint32_t hw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t* p0 = reinterpret_cast<const uint32_t*>(&pv[k][0]);
          f2_t acc = bf2_to_f2(p0[i]);
#pragma unroll
          for (int t = 1; t < T; ++t)
            acc = f2_add(acc, bf2_to_f2(reinterpret_cast<const uint32_t*>(&pv[k][t])[i]));
          float al, ah;
          f2_split(acc, al, ah);
          acc = f2(((keep >> (2 * i)) & 1u) ? al : 0.f, ((keep >> (2 * i + 1)) & 1u) ? ah : 0.f);
          hw[i] = residual_bf2(bf2_to_f2(reinterpret_cast<const uint32_t*>(&rv[k])[i]), acc, shi, slo);
          hf[k][i] = bf2_to_f2(hw[i]);  // the norm reads the stored (rounded) value
          s2 = LN ? f2_add(s2, hf[k][i]) : f2_fma(hf[k][i], hf[k][i], s2);
        }
        hout = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      } else {
        float acc[EV], tmp[EV], rs[EV], hv[EV];
        V::unpack(pv[k][0], acc);
#pragma unroll
        for (int t = 1; t < T; ++t) {
          V::unpack(pv[k][t], tmp);
#pragma unroll
          for (int e = 0; e < EV; ++e) acc[e] += tmp[e];
        }
        V::unpack(rv[k], rs);
#pragma unroll
        for (int e = 0; e < EV; ++e) hv[e] = rs[e] + (((keep >> e) & 1u) ? acc[e] * a.scale : 0.f);
        hout = V::pack(hv);
        hp[k] = hout;
#pragma unroll
        for (int e = 0; e < EV; ++e) s += LN ? hv[e] : hv[e] * hv[e];
      }
      st_stream(reinterpret_cast<Act*>(a.h) + r * (int64_t)a.H + (int64_t)v * EV, hout);
      if (a.mask) st_mask<EV>(a.mask + r * (int64_t)a.H + (int64_t)v * EV, keep);
    }
  }
  if constexpr (EV == 8) {
    float lo, hi;
    f2_split(s2, lo, hi);
    s = lo + hi;
  }

  // ---- row statistics ------------------------------------------------------
  float* rred = red + rg * 2 * (tpr >> 5);
  float sv[1] = {s};
  row_allreduce<1>(sv, tpr, lr, 1 + rg, rred, 0);
  float mu = 0.f, rstd;
  if constexpr (LN) {
    mu = sv[0] / a.Hf;
    float q = 0.f;
    f2_t q2 = f2(0.f, 0.f);
    const f2_t mu2 = f2(mu, mu);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (lr + k * tpr < a.nvec) {
        if constexpr (EV == 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const f2_t dd = f2_sub(hf[k][i], mu2);
            q2 = f2_fma(dd, dd, q2);
          }
        } else {
          float hr[EV];
          V::unpack(hp[k], hr);
#pragma unroll
          for (int e = 0; e < EV; ++e) {
            const float d = hr[e] - mu;
            q += d * d;
          }
        }
      }
    }
    if constexpr (EV == 8) {
      float lo, hi;
      f2_split(q2, lo, hi);
      q = lo + hi;
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
      uint4 yout;
      if constexpr (EV == 8) {
        const f2_t r2 = f2(rstd, rstd), mu2 = f2(mu, mu);
        const uint4 gw = sgb[v];
        const uint4 bw = LN ? sgb[a.nvec + v] : gw;
        uint32_t yw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const f2_t g = bf2_to_f2(reinterpret_cast<const uint32_t*>(&gw)[i]);
          f2_t yv;
          if constexpr (LN)
            yv = f2_fma(g, f2_mul(f2_sub(hf[k][i], mu2), r2),
                        bf2_to_f2(reinterpret_cast<const uint32_t*>(&bw)[i]));
          else
            yv = f2_mul(g, f2_mul(hf[k][i], r2));
          yw[i] = f2_to_bf2(yv);
        }
        yout = make_uint4(yw[0], yw[1], yw[2], yw[3]);
      } else {
        float gm[EV], hr[EV], yv[EV];
        V::unpack(sgb[v], gm);
        V::unpack(hp[k], hr);
        if constexpr (LN) {
          float bt[EV];
          V::unpack(sgb[a.nvec + v], bt);
#pragma unroll
          for (int e = 0; e < EV; ++e) yv[e] = gm[e] * ((hr[e] - mu) * rstd) + bt[e];
        } else {
#pragma unroll
          for (int e = 0; e < EV; ++e) yv[e] = gm[e] * (hr[e] * rstd);
        }
        yout = V::pack(yv);
      }
      st_keep(reinterpret_cast<Act*>(a.y) + r * (int64_t)a.H + (int64_t)v * EV, yout);
    }
  }
  if (lr == 0) {
    a.rstd[r] = rstd;
    if constexpr (LN) a.mean[r] = mu;
  }
}

}  // namespace spf
