// launch.h -- host-side launch helpers and the internal launcher table of
// libspfuse (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spfuse.h"
#include "common.cuh"
#include "tma.cuh"

namespace spf {

// The allocation-free backward keeps its partial rows in a fixed array of
// SP_NOALLOC_SCRATCH_BYTES and refuses problems whose workspace exceeds it.
inline bool noalloc_scratch_fits(size_t workspace_bytes) {
  return workspace_bytes <= (size_t)SP_NOALLOC_SCRATCH_BYTES;
}

// The TMA-fed kernels prefetch their first ring stages into L2 before the
// grid-dependency wait: as many stages as it takes to reach this many bytes
// per CTA (at least one), about what keeps one SM's share of HBM busy.
constexpr size_t kPrefetchBytes = 48 * 1024;
inline int prefetch_stages(size_t stage_bytes) {
  return (int)((kPrefetchBytes + stage_bytes - 1) / stage_bytes);
}

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel in the stream drains; it does not read
// memory before griddepcontrol.wait, so stream order is kept.
template <typename... KArgs, typename... Args>
inline cudaError_t pdl_launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Dynamic shared memory above this needs the per-kernel opt-in (the default
// limit is 48 KB including the kernels' small static shared arrays).
constexpr size_t kSmemOptInThreshold = 46 * 1024;

// Row kernel shape: threads per row, 16-byte vectors per thread, block size.
struct RowShape {
  int tpr;
  int vpt;
  int block;
};

// Forward launchers, one translation unit per (activation, norm); T in 1..8
// and VPT in 1..4 are compile-time.
cudaError_t launch_fwd_bf16_rms(const FwdArgs& a, int T, const RowShape& s, dim3 grid, cudaStream_t st);
cudaError_t launch_fwd_bf16_ln(const FwdArgs& a, int T, const RowShape& s, dim3 grid, cudaStream_t st);
cudaError_t launch_fwd_f32_rms(const FwdArgs& a, int T, const RowShape& s, dim3 grid, cudaStream_t st);
cudaError_t launch_fwd_f32_ln(const FwdArgs& a, int T, const RowShape& s, dim3 grid, cudaStream_t st);

// Backward launchers (VPT in 1..4) and their occupancy (CTAs per SM).
cudaError_t launch_bwd(int dtype, bool ln, const BwdArgs& a, const RowShape& s, dim3 grid,
                       size_t smem, cudaStream_t st);
int bwd_max_active_clusters(int dtype, bool ln, const RowShape& s, size_t smem);
cudaError_t launch_colsum(const float* ws, int nparts, int H, bool ln, float* dgamma,
                          float* dbeta, bool accumulate, cudaStream_t st);

// TMA-fed backward (bf16, H % 16 == 0): shared-memory ring layout and shape.
// Block sizes the TMA backward is compiled for: 15 consumer warps + producer
// (128 registers), or two 8-warp row groups + producer (96 registers, up to
// 3 vectors a thread) for rows of 256 threads.
constexpr int kBwdTmaNarrow = 512;
constexpr int kBwdTmaMid = 544;

struct BwdTmaPlan {
  RowShape shape;
  size_t smem;
  int nthr;  // kBwdTmaNarrow or kBwdTmaMid
  BwdTmaLayout layout;
};
bool plan_bwd_tma(int64_t H, bool ln, bool has_dh, bool has_mask, int max_smem, int64_t rows_per_cta,
                  BwdTmaPlan* p);
cudaError_t launch_bwd_tma(bool ln, const BwdArgs& a, const BwdTmaPlan& p, dim3 grid, cudaStream_t st);
cudaError_t launch_bwd_tma_rms(const BwdArgs& a, const BwdTmaPlan& p, dim3 grid, cudaStream_t st);
cudaError_t launch_bwd_tma_ln(const BwdArgs& a, const BwdTmaPlan& p, dim3 grid, cudaStream_t st);

// TMA-fed forward (bf16, rows short enough for a two-stage ring).
// Block sizes the TMA forward is compiled for: 16 consumer warps + producer
// (registers for T up to 8), or 27 + producer (72 registers, T <= 4).
constexpr int kFwdTmaDeep = 544;
constexpr int kFwdTmaWide = 896;
constexpr int kFwdTmaWideMaxT = 4;

struct FwdTmaPlan {
  RowShape shape;
  size_t smem;
  int nthr;     // kFwdTmaDeep or kFwdTmaWide
  bool chunked;  // stages of one column chunk of one row
  FwdTmaLayout layout;
};
bool plan_fwd_tma(int64_t H, int T, bool ln, int max_smem, int64_t rows, int sms, FwdTmaPlan* p);
cudaError_t launch_fwd_tma_rms(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid, cudaStream_t st);
cudaError_t launch_fwd_tma_ln(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid, cudaStream_t st);
cudaError_t launch_fwd_tma_rms_ch(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid, cudaStream_t st);
cudaError_t launch_fwd_tma_ln_ch(const FwdArgs& a, int T, const FwdTmaPlan& p, dim3 grid, cudaStream_t st);

cudaError_t launch_layout(bool to_hp, const void* in, void* out, int64_t N, int64_t H, int32_t T,
                          int elem_bytes, cudaStream_t stream);

}  // namespace spf
