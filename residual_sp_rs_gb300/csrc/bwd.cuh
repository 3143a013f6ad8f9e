// bwd.cuh -- backward of the SP region (norm backward, residual-add and
// dropout backward) and the first pass of the dgamma/dbeta reduction.
//
// A persistent-style grid: CTA b owns the contiguous rows
// [b*rows_per_cta, (b+1)*rows_per_cta); its row groups walk those rows one
// row at a time.  A thread owns the same columns on every row, so its
// dgamma/dbeta contributions accumulate in registers across rows.  At the end
// the CTA adds its row groups' sums in row-group order into shared memory;
// the 8 CTAs of a thread-block cluster then add their sums through
// distributed shared memory in rank order and write one fp32 partial row per
// statistic per cluster; sp_colsum_kernel adds the partial rows in cluster
// order.  The result is bit-identical from run to run.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace spf {

namespace cg = cooperative_groups;

constexpr int kBwdCluster = 8;  // CTAs per thread-block cluster in the backward

// The compiler must not keep unpacked copies of these registers alive across
// the row reduction; re-unpacking after it is cheaper than the registers.
__device__ __forceinline__ void opaque(uint4& v) {
  asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
}

template <typename Act, bool LN, int VPT>
__global__ void __cluster_dims__(kBwdCluster, 1, 1) __launch_bounds__(512)
    sp_bwd_kernel(const BwdArgs a) {
  using V = Act16<Act>;
  constexpr int EV = V::EV;
  constexpr int NS = LN ? 2 : 1;  // row sums needed: mean(g*xhat) (+ mean(g))
  __shared__ float red[2 * 32 * 2];
  extern __shared__ float colacc[];  // [NS][H] CTA column sums, then gamma vectors [nvec]
  uint4* sgam = reinterpret_cast<uint4*>(colacc + NS * a.H);

  const int tpr = a.tpr;
  const int rg = threadIdx.x / tpr;
  const int lr = threadIdx.x - rg * tpr;
  const int rpc = blockDim.x / tpr;
  const int64_t r0 = (int64_t)blockIdx.x * a.rows_per_cta;
  const int64_t r1 = min(a.rows, r0 + a.rows_per_cta);

  grid_dep_wait();
  grid_dep_launch_dependents();

  for (int i = threadIdx.x; i < a.nvec; i += blockDim.x)
    sgam[i] = ld_cached(reinterpret_cast<const Act*>(a.gamma) + i * EV);
  __syncthreads();

  float dg[VPT][EV];
  float db[LN ? VPT : 1][EV];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
#pragma unroll
    for (int e = 0; e < EV; ++e) {
      dg[k][e] = 0.f;
      if constexpr (LN) db[k][e] = 0.f;
    }
  }

  float* rred = red + rg * 2 * (tpr >> 5) * NS;
  int slot = 0;
  for (int64_t r = r0 + rg; r < r1; r += rpc) {
    const int64_t ro = r * (int64_t)a.H;
    uint4 dyv[VPT], dhv[VPT], hv[VPT];
    uint32_t mk[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lr + k * tpr;
      if (v < a.nvec) {
        const int64_t o = ro + (int64_t)v * EV;
        dyv[k] = ld_stream(reinterpret_cast<const Act*>(a.dy) + o);
        hv[k] = ld_stream(reinterpret_cast<const Act*>(a.h) + o);
        dhv[k] = a.dh ? ld_stream(reinterpret_cast<const Act*>(a.dh) + o) : make_uint4(0u, 0u, 0u, 0u);
        if (a.mask) {
          mk[k] = ld_mask<EV>(a.mask + o);
        } else if (a.regen) {  // the forward's keep bits, from the same generator
          const uint64_t g0 = (uint64_t)((a.grow0 + r) * (int64_t)a.H + (int64_t)v * EV);
          mk[k] = keep_bits4(g0 >> 2, a.keys, a.thr);
          if constexpr (EV == 8) mk[k] |= keep_bits4((g0 >> 2) + 1, a.keys, a.thr) << 4;
        } else {
          mk[k] = (1u << EV) - 1u;
        }
      }
    }
    const float rstd = __ldcs(a.rstd + r);
    const float mu = LN ? __ldcs(a.mean + r) : 0.f;

    // pass 1: the row sums of g*xhat (and g)
    float sums[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) sums[i] = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (lr + k * tpr < a.nvec) {
        float dyf[EV], hf[EV], gm[EV];
        V::unpack(dyv[k], dyf);
        V::unpack(hv[k], hf);
        V::unpack(sgam[lr + k * tpr], gm);
#pragma unroll
        for (int e = 0; e < EV; ++e) {
          const float g = gm[e] * dyf[e];
          sums[0] += g * ((hf[e] - mu) * rstd);
          if constexpr (LN) sums[1] += g;
        }
      }
    }
    row_allreduce<NS>(sums, tpr, lr, 1 + rg, rred, slot);
    slot ^= 1;
    const float c_gx = sums[0] / a.Hf;
    const float c_g = LN ? sums[NS - 1] / a.Hf : 0.f;

    // pass 2: input gradients, mask-gated gradient of the partials, dgamma/dbeta
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lr + k * tpr;
      if (v < a.nvec) {
        opaque(dyv[k]);
        opaque(hv[k]);
        float dyf[EV], hf[EV], gm[EV], dhf[EV], dres[EV], dsum[EV];
        V::unpack(dyv[k], dyf);
        V::unpack(hv[k], hf);
        V::unpack(dhv[k], dhf);
        V::unpack(sgam[v], gm);
#pragma unroll
        for (int e = 0; e < EV; ++e) {
          const float xh = (hf[e] - mu) * rstd;
          const float g = gm[e] * dyf[e];
          dres[e] = rstd * (g - c_g - xh * c_gx) + dhf[e];
          dsum[e] = ((mk[k] >> e) & 1u) ? dres[e] * a.scale : 0.f;
          dg[k][e] += dyf[e] * xh;
          if constexpr (LN) db[k][e] += dyf[e];
        }
        const int64_t o = ro + (int64_t)v * EV;
        st_stream(reinterpret_cast<Act*>(a.d_res) + o, V::pack(dres));
        st_stream(reinterpret_cast<Act*>(a.d_sum) + o, V::pack(dsum));
      }
    }
  }

  // ---- CTA column sums in row-group order ---------------------------------
  for (int q = 0; q < rpc; ++q) {
    if (rg == q) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lr + k * tpr;
        if (v < a.nvec) {
#pragma unroll
          for (int e = 0; e < EV; ++e) {
            const int c = v * EV + e;
            colacc[c] = (q == 0) ? dg[k][e] : colacc[c] + dg[k][e];
            if constexpr (LN) colacc[a.H + c] = (q == 0) ? db[k][e] : colacc[a.H + c] + db[k][e];
          }
        }
      }
    }
    __syncthreads();
  }

  // ---- cluster column sums over distributed shared memory -----------------
  // CTA rank q of the cluster adds column slice q of all kBwdCluster CTAs'
  // sums, in rank order, and writes it to the cluster's partial row; the
  // second pass then reads one row per cluster instead of one per CTA.
  cg::cluster_group cl = cg::this_cluster();
  cl.sync();
  const int q = (int)cl.block_rank();
  const int n4 = a.H >> 2;
  const int per = (n4 + kBwdCluster - 1) / kBwdCluster;
  const int c_end = min(n4, (q + 1) * per);
  const int64_t cluster_id = blockIdx.x / kBwdCluster;
#pragma unroll
  for (int st = 0; st < NS; ++st) {
    float4* out = reinterpret_cast<float4*>(a.ws + ((int64_t)st * a.nparts + cluster_id) * a.H);
    for (int c4 = q * per + (int)threadIdx.x; c4 < c_end; c4 += blockDim.x) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int p = 0; p < kBwdCluster; ++p) {
        const float4 w =
            reinterpret_cast<const float4*>(cl.map_shared_rank(colacc + st * a.H, p))[c4];
        s.x += w.x;
        s.y += w.y;
        s.z += w.z;
        s.w += w.w;
      }
      __stcg(out + c4, s);
    }
  }
  cl.sync();  // keep this CTA's shared memory alive until every peer has read it
}

// Second pass: dgamma[c] (and dbeta[c]) = the sum over partial rows
// p = 0..nparts-1.  blockDim (32, 32): x picks a float4 column of a 32-column
// group, y a stride class of partial rows (p = y, y+32, ...).  Each thread
// issues all its loads (up to 8 per round) before adding, then the 32 stride
// sums are added pairwise (y + 16, 8, 4, 2, 1).  The order is fixed, so the
// result is bit-identical from run to run.  With `accumulate` the sum is added
// to what dgamma/dbeta hold (the earlier chunks of a row range), else it
// replaces it.
__global__ void __launch_bounds__(1024) sp_colsum_kernel(const float* ws, int nparts, int H,
                                                         float* dgamma, float* dbeta, int accumulate) {
  __shared__ float4 part[32][32];
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int stat = blockIdx.y;
  const float* src = ws + (int64_t)stat * nparts * H;
  float* dst = stat ? dbeta : dgamma;
  const int c4 = blockIdx.x * 32 + threadIdx.x;
  const int n4 = H / 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c4 < n4) {
    for (int p0 = threadIdx.y; p0 < nparts; p0 += 32 * 8) {
      float4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = p0 + 32 * u;
        w[u] = p < nparts ? __ldcg(reinterpret_cast<const float4*>(src + (int64_t)p * H) + c4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x += w[u].x;
        acc.y += w[u].y;
        acc.z += w[u].z;
        acc.w += w[u].w;
      }
    }
  }
  // the 32 stride sums of a column, added pairwise in a fixed tree
  part[threadIdx.y][threadIdx.x] = acc;
#pragma unroll
  for (int half = 16; half > 0; half >>= 1) {
    __syncthreads();
    if (threadIdx.y < half) {
      const float4 w = part[threadIdx.y + half][threadIdx.x];
      acc.x += w.x;
      acc.y += w.y;
      acc.z += w.z;
      acc.w += w.w;
      part[threadIdx.y][threadIdx.x] = acc;
    }
  }
  if (threadIdx.y == 0 && c4 < n4) {
    float4* d4 = reinterpret_cast<float4*>(dst) + c4;
    if (accumulate) {
      const float4 o = *d4;
      acc = make_float4(o.x + acc.x, o.y + acc.y, o.z + acc.z, o.w + acc.w);
    }
    *d4 = acc;
  }
}

}  // namespace spf
