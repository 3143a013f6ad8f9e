// layout.cu -- sp2hp / hp2sp (LLM Infra Atlas "03 · Sequence Parallelism",
// §5): the all-to-all between the sequence-split layout [N/T, H] per rank
// and the hidden-split layout [N, H/T] per rank, as one permutation copy on
// a GPU that holds all T rank buffers.
//
// Each thread moves kLayoutVPT 16-byte vectors, issuing all loads before any
// store.
// sp2hp walks the INPUT in order (coalesced reads; a warp's writes stay
// inside one destination chunk of H/T elements except at chunk edges);
// hp2sp walks the OUTPUT in order.  Index math is 32-bit when the vector
// count allows it.  Before the grid-dependency wait, thread 0 of each CTA
// starts bringing the CTA's input bytes into L2 (a hint: the loads after the
// wait read whatever the previous kernel wrote), so in a stream the reads
// overlap the previous kernel's tail.
#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace spf {

namespace {

// 128-thread CTAs: sp2hp of 12.6 MB 2.70 instead of 3.08 us with 256 (the
// same at 268 MB).
constexpr int kLayoutThreads = 128;
constexpr int kLayoutVPT = 2;  // 2-4 measure alike; 8 (fewer CTAs) is slower

// nv: vectors per [N,H] row; ncv: vectors per H/T chunk.
template <bool TO_HP, typename Idx>
__global__ void __launch_bounds__(kLayoutThreads)
    sp_layout_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, Idx total, Idx N,
                     Idx nv, Idx ncv) {
  const Idx first = (Idx)blockIdx.x * (kLayoutThreads * kLayoutVPT);  // this CTA's walk
  if (threadIdx.x == 0) {
    const Idx last = min(total, first + (Idx)(kLayoutThreads * kLayoutVPT));  // exclusive
    if (TO_HP) {
      l2_prefetch(in + first, (uint32_t)((last - first) * 16));
    } else {
      // the rows n0..n1 of each rank's plane r: (r*N + n)*ncv .. + ncv
      const Idx n0 = first / nv, n1 = (last - 1) / nv;
      const Idx T = nv / ncv;
      for (Idx r = 0; r < T; ++r)
        l2_prefetch(in + (r * N + n0) * ncv, (uint32_t)((n1 - n0 + 1) * ncv * 16));
    }
  }
  grid_dep_wait();
  grid_dep_launch_dependents();
  const Idx base = first + threadIdx.x;
  uint4 buf[kLayoutVPT];
  Idx dst[kLayoutVPT];
#pragma unroll
  for (int k = 0; k < kLayoutVPT; ++k) {
    const Idx i = base + (Idx)k * kLayoutThreads;  // position in the walked ([N,H]) order
    if (i < total) {
      const Idx n = i / nv;
      const Idx v = i - n * nv;
      const Idx r = v / ncv;
      const Idx c = v - r * ncv;
      const Idx o = (r * N + n) * ncv + c;  // position in [T][N][H/T]
      if (TO_HP) {
        buf[k] = ld_stream(in + i);
        dst[k] = o;
      } else {
        buf[k] = ld_stream(in + o);
        dst[k] = i;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kLayoutVPT; ++k) {
    const Idx i = base + (Idx)k * kLayoutThreads;
    if (i < total) st_stream(out + dst[k], buf[k]);
  }
}

template <bool TO_HP>
cudaError_t launch_layout_t(const void* in, void* out, int64_t N, int64_t H, int32_t T,
                            int elem_bytes, cudaStream_t stream) {
  const int ev = 16 / elem_bytes;
  const int64_t nv = H / ev;
  const int64_t ncv = (H / T) / ev;
  const int64_t total = N * nv;
  if (total == 0) return cudaSuccess;
  const int64_t per_block = (int64_t)kLayoutThreads * kLayoutVPT;
  const dim3 grid((unsigned)((total + per_block - 1) / per_block));
  const dim3 block(kLayoutThreads);
  if (total < ((int64_t)1 << 31) - per_block) {
    return pdl_launch(sp_layout_kernel<TO_HP, uint32_t>, grid, block, 0, stream,
                      (const uint4*)in, (uint4*)out, (uint32_t)total, (uint32_t)N, (uint32_t)nv,
                      (uint32_t)ncv);
  }
  return pdl_launch(sp_layout_kernel<TO_HP, uint64_t>, grid, block, 0, stream, (const uint4*)in,
                    (uint4*)out, (uint64_t)total, (uint64_t)N, (uint64_t)nv, (uint64_t)ncv);
}

}  // namespace

cudaError_t launch_layout(bool to_hp, const void* in, void* out, int64_t N, int64_t H, int32_t T,
                          int elem_bytes, cudaStream_t stream) {
  return to_hp ? launch_layout_t<true>(in, out, N, H, T, elem_bytes, stream)
               : launch_layout_t<false>(in, out, N, H, T, elem_bytes, stream);
}

}  // namespace spf
