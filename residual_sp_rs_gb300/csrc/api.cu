// api.cu -- the C ABI of libspfuse: argument validation, kernel-shape
// selection and launches.  Declarations and the contract of every entry
// point are in include/spfuse.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/spfuse.h"
#include "launch.h"

namespace spf {
namespace {

constexpr int kMaxFwdTPR = 512;
constexpr int kMaxVPT = 4;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int elem_bytes(int dtype) { return dtype == SP_BF16 ? 2 : 4; }

// Test hook: when SPFUSE_FAIL_LAUNCH is set in the environment, every launch
// reports a CUDA failure without touching the GPU, so error propagation can be
// exercised on a machine with or without a device.
bool inject_launch_failure() {
  static const bool on = std::getenv("SPFUSE_FAIL_LAUNCH") != nullptr;
  return on;
}

// Test hooks for the bounded waits, read once per process: SPFUSE_TEST_WAIT_NS
// shortens the limit of every mbarrier wait (nanoseconds) and
// SPFUSE_TEST_DROP_STAGE makes the producer of CTA 0 of the TMA-fed kernels
// skip that ring stage, so the waits on it run out and the kernels take
// their timeout path (no fault, no hang: every wait returns).
struct WaitHooks {
  uint64_t wait_ns;
  int32_t drop_stage;
};

const WaitHooks& wait_hooks() {
  static const WaitHooks h = [] {
    WaitHooks w{kWaitNs, -1};
    if (const char* e = std::getenv("SPFUSE_TEST_WAIT_NS")) w.wait_ns = std::strtoull(e, nullptr, 10);
    if (const char* e = std::getenv("SPFUSE_TEST_DROP_STAGE")) w.drop_stage = std::atoi(e);
    return w;
  }();
  return h;
}

// The CUDA error behind the last SP_ERR_CUDA on this host thread.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

sp_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return SP_OK;
  g_last_cuda_error = e;
  return SP_ERR_CUDA;
}

struct Problem {
  int T, j, nshards, dtype, norm;
  int64_t S, B, H, R, rows;
  int ev, nvec;
};

// Checks the descriptor (not the pointers) and derives the row counts.
sp_status_t check_desc(const sp_rs_desc_t* d, Problem* pr) {
  if (!d) return SP_ERR_INVALID_ARG;
  if (d->dtype != SP_F32 && d->dtype != SP_BF16) return SP_ERR_DTYPE;
  if (d->norm != SP_RMSNORM && d->norm != SP_LAYERNORM) return SP_ERR_DTYPE;
  const int nsh = d->nshards == 0 ? 1 : d->nshards;
  if (d->T < 1 || d->T > kMaxT || d->j < 0 || d->j >= d->T || nsh < 1 || d->j + nsh > d->T ||
      d->reserved != 0)
    return SP_ERR_INVALID_ARG;
  if (!(d->p >= 0.0f && d->p < 1.0f)) return SP_ERR_INVALID_ARG;
  if (!(d->eps > 0.0f) || !std::isfinite(d->eps)) return SP_ERR_INVALID_ARG;
  if (!aligned(d->status, 4)) return SP_ERR_ALIGN;
  if (d->S < 0 || d->B < 0 || d->H <= 0) return SP_ERR_SHAPE;
  if (d->S % d->T != 0) return SP_ERR_SHAPE;
  const int ev = 16 / elem_bytes(d->dtype);
  if (d->H % ev != 0) return SP_ERR_SHAPE;
  // row length limit of the register-resident row kernels
  if (d->H / ev > (int64_t)kMaxFwdTPR * kMaxVPT) return SP_ERR_SHAPE;
  // every element index must fit comfortably in int64
  if (d->S > 0 && d->B > 0 && (d->S > ((int64_t)1 << 40) / d->B || d->S * d->B > ((int64_t)1 << 46) / d->H))
    return SP_ERR_SHAPE;
  pr->T = d->T;
  pr->j = d->j;
  pr->nshards = nsh;
  pr->dtype = d->dtype;
  pr->norm = d->norm;
  pr->S = d->S;
  pr->B = d->B;
  pr->H = d->H;
  pr->R = (d->S / d->T) * d->B;
  pr->rows = pr->R * nsh;
  pr->ev = ev;
  pr->nvec = (int)(d->H / ev);
  return SP_OK;
}

// Largest VPT the forward keeps in registers without spilling, by T.
int fwd_vpt_cap(int T) { return T <= 2 ? 4 : (T <= 4 ? 3 : 2); }

RowShape row_shape(int nvec, int vpt_cap) {
  int tpr = 32;
  while (tpr < kMaxFwdTPR && (nvec + tpr - 1) / tpr > vpt_cap) tpr *= 2;
  RowShape s;
  s.tpr = tpr;
  s.vpt = (nvec + tpr - 1) / tpr;
  s.block = tpr >= 256 ? tpr : 256;
  return s;
}

RowShape bwd_row_shape(const Problem& pr) { return row_shape(pr.nvec, pr.ev == 8 ? 3 : 4); }

struct BwdPlan {
  bool tma;    // TMA-fed kernel (else the register kernel with cluster partials)
  BwdTmaPlan tp;
  RowShape shape;
  size_t smem;
  int64_t rows_per_cta;
  int ctas;    // register kernel: a multiple of the cluster size
  int nparts;  // partial rows per statistic (CTAs or clusters)
  size_t ws_bytes;
};

// has_dh / has_mask only shape the TMA ring; the choice of kernel and the
// workspace size are decided with both present, so the workspace query and
// the call always agree.
// The TMA-fed backward on a device with `sms` multiprocessors and `optin`
// bytes of opt-in shared memory per block, when it applies (bf16 and a ring
// that fits): one CTA per SM over contiguous rows, one partial row each.
bool plan_bwd_tma_for(const Problem& pr, bool has_dh, bool has_mask, int sms, int optin, BwdPlan* pl) {
  const bool ln = pr.norm == SP_LAYERNORM;
  if (pr.dtype != SP_BF16) return false;
  const int64_t ctas = pr.rows < sms ? (pr.rows > 0 ? pr.rows : 1) : sms;
  const int64_t rpc = pr.rows > 0 ? (pr.rows + ctas - 1) / ctas : 1;
  BwdTmaPlan probe;
  if (!plan_bwd_tma(pr.H, ln, true, true, optin, rpc, &probe) ||
      !plan_bwd_tma(pr.H, ln, has_dh, has_mask, optin, rpc, &pl->tp))
    return false;
  pl->tma = true;
  pl->rows_per_cta = rpc;
  pl->ctas = pr.rows > 0 ? (int)((pr.rows + pl->rows_per_cta - 1) / pl->rows_per_cta) : 0;
  pl->nparts = pl->ctas;
  pl->ws_bytes = (size_t)(ctas > 0 ? ctas : 1) * (size_t)pr.H * sizeof(float) * (ln ? 2 : 1);
  return true;
}

sp_status_t plan_bwd(const Problem& pr, bool has_dh, bool has_mask, BwdPlan* pl) {
  const bool ln = pr.norm == SP_LAYERNORM;
  pl->tma = false;
  if (pr.dtype == SP_BF16) {
    int dev = 0, sms = 0, optin = 0;
    cudaError_t qe = cudaGetDevice(&dev);
    if (qe == cudaSuccess) qe = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (qe == cudaSuccess)
      qe = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (qe != cudaSuccess) return from_cuda(qe);
    if (plan_bwd_tma_for(pr, has_dh, has_mask, sms, optin, pl)) return SP_OK;
  }
  pl->tma = false;
  pl->shape = bwd_row_shape(pr);
  // CTA column sums, then the gamma vectors
  pl->smem = (size_t)(ln ? 2 : 1) * (size_t)pr.H * sizeof(float) + (size_t)pr.nvec * 16;
  const int clusters = bwd_max_active_clusters(pr.dtype, ln, pl->shape, pl->smem);
  if (clusters < 1) return SP_ERR_CUDA;
  const int cluster = 8;
  const int rpc = pl->shape.block / pl->shape.tpr;
  // as many CTAs as are resident at once, but at least one row per row group
  int64_t want = (pr.rows + rpc - 1) / rpc;
  int64_t cap = (int64_t)clusters * cluster;
  int64_t ctas = want < cap ? want : cap;
  ctas = ((ctas + cluster - 1) / cluster) * cluster;
  if (ctas < cluster) ctas = cluster;
  pl->rows_per_cta = pr.rows > 0 ? (pr.rows + ctas - 1) / ctas : 1;
  pl->ctas = (int)ctas;
  pl->nparts = (int)(ctas / cluster);
  pl->ws_bytes = (size_t)pl->nparts * (size_t)pr.H * sizeof(float) * (ln ? 2 : 1);
  return SP_OK;
}

// The forward over rows [row_begin, row_begin + row_count) of the call's
// nshards*R rows (all of them unless `ranged`).  Per-row arguments address
// the call's row 0; the partials and the dropout mask follow the global row
// index, so a range computes exactly what the full call computes there.
sp_status_t fwd_impl(const sp_rs_desc_t* desc, bool ranged, int64_t row_begin, int64_t row_count,
                     const void* const* partials, const void* residual, const void* gamma,
                     const void* beta, void* h_out, void* y_out, uint8_t* mask_out,
                     float* rstd_out, float* mean_out, sp_stream_t stream) {
  Problem pr;
  sp_status_t st = check_desc(desc, &pr);
  if (st != SP_OK) return st;
  const bool ln = pr.norm == SP_LAYERNORM;
  if (!ranged) {
    row_begin = 0;
    row_count = pr.rows;
  } else if (row_begin < 0 || row_count < 0 || row_begin > pr.rows || row_count > pr.rows - row_begin) {
    return SP_ERR_INVALID_ARG;
  }
  if (row_count == 0) return SP_OK;  // nothing to read or write
  if (!partials || !residual || !gamma || !h_out || !y_out || !rstd_out) return SP_ERR_INVALID_ARG;
  if (ln && (!beta || !mean_out)) return SP_ERR_INVALID_ARG;
  for (int t = 0; t < pr.T; ++t) {
    if (!partials[t]) return SP_ERR_INVALID_ARG;
    if (!aligned(partials[t], 16)) return SP_ERR_ALIGN;
  }
  // the range's first row of every per-row argument
  const int64_t rowb = pr.H * elem_bytes(pr.dtype);
  residual = static_cast<const char*>(residual) + row_begin * rowb;
  h_out = static_cast<char*>(h_out) + row_begin * rowb;
  y_out = static_cast<char*>(y_out) + row_begin * rowb;
  if (mask_out) mask_out += row_begin * pr.H;
  rstd_out += row_begin;
  if (ln) mean_out += row_begin;
  if (!aligned(residual, 16) || !aligned(gamma, 16) || !aligned(h_out, 16) || !aligned(y_out, 16) ||
      (ln && !aligned(beta, 16)) || (mask_out && !aligned(mask_out, 16)) || !aligned(rstd_out, 4) ||
      (ln && !aligned(mean_out, 4)))
    return SP_ERR_ALIGN;

  FwdArgs a = {};
  for (int t = 0; t < pr.T; ++t) a.P[t] = partials[t];
  a.residual = residual;
  a.gamma = gamma;
  a.beta = ln ? beta : nullptr;
  a.h = h_out;
  a.y = y_out;
  a.mask = mask_out;
  a.rstd = rstd_out;
  a.mean = ln ? mean_out : nullptr;
  a.rows = row_count;
  a.grow0 = (int64_t)pr.j * pr.R + row_begin;
  a.H = (int32_t)pr.H;
  a.nvec = pr.nvec;
  a.thr = (uint32_t)std::floor((double)desc->p * 4294967296.0);
  // Philox round keys: the seed's two words advanced by the Weyl increments
  for (int i = 0; i < 10; ++i) {
    a.keys.rk[2 * i] = (uint32_t)desc->seed + (uint32_t)i * 0x9E3779B9u;
    a.keys.rk[2 * i + 1] = (uint32_t)(desc->seed >> 32) + (uint32_t)i * 0xBB67AE85u;
  }
  const double scale = 1.0 / (1.0 - (double)desc->p);
  a.scale = (float)scale;
  a.scale_lo = (float)(scale - (double)a.scale);
  a.eps = desc->eps;
  a.Hf = (float)pr.H;
  a.dropout = desc->p > 0.0f ? 1 : 0;
  a.dyadic_scale = a.scale_lo == 0.0f ? 1 : 0;
  a.status = desc->status;
  a.wait_ns = wait_hooks().wait_ns;
  a.drop_stage = wait_hooks().drop_stage;

  if (inject_launch_failure()) return SP_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (pr.dtype == SP_BF16) {
    int dev = 0, sms = 0, optin = 0;
    cudaError_t qe = cudaGetDevice(&dev);
    if (qe == cudaSuccess) qe = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (qe == cudaSuccess)
      qe = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (qe != cudaSuccess) return from_cuda(qe);
    FwdTmaPlan tp;
    if (plan_fwd_tma(pr.H, pr.T, ln, optin, row_count, sms, &tp)) {
      a.tpr = tp.shape.tpr;
      const dim3 grid((unsigned)((row_count + tp.layout.rows_per_cta - 1) / tp.layout.rows_per_cta));
      return from_cuda(ln ? launch_fwd_tma_ln(a, pr.T, tp, grid, cs)
                          : launch_fwd_tma_rms(a, pr.T, tp, grid, cs));
    }
  }
  const RowShape s = row_shape(pr.nvec, fwd_vpt_cap(pr.T));
  a.tpr = s.tpr;
  const int rpc = s.block / s.tpr;
  const dim3 grid((unsigned)((row_count + rpc - 1) / rpc));
  cudaError_t e;
  if (pr.dtype == SP_BF16)
    e = ln ? launch_fwd_bf16_ln(a, pr.T, s, grid, cs) : launch_fwd_bf16_rms(a, pr.T, s, grid, cs);
  else
    e = ln ? launch_fwd_f32_ln(a, pr.T, s, grid, cs) : launch_fwd_f32_rms(a, pr.T, s, grid, cs);
  return from_cuda(e);
}

// The backward over rows [row_begin, row_begin + row_count) of the call's
// nshards*R rows (all of them unless `ranged`).  Per-row arguments address
// the call's row 0; the regenerated mask follows the global row index.
// dgamma/dbeta receive the range's sums, added to what they hold when
// `accumulate` is set.
sp_status_t bwd_impl(const sp_rs_desc_t* desc, bool ranged, int64_t row_begin, int64_t row_count,
                     bool accumulate, const void* dy, const void* dh_out, const void* h_saved,
                     const void* gamma, const uint8_t* mask, const float* rstd, const float* mean,
                     void* d_residual, void* d_sum, float* dgamma, float* dbeta, void* workspace,
                     size_t workspace_bytes, sp_stream_t stream) {
  Problem pr;
  sp_status_t st = check_desc(desc, &pr);
  if (st != SP_OK) return st;
  const bool ln = pr.norm == SP_LAYERNORM;
  if (!ranged) {
    row_begin = 0;
    row_count = pr.rows;
  } else if (row_begin < 0 || row_count < 0 || row_begin > pr.rows || row_count > pr.rows - row_begin) {
    return SP_ERR_INVALID_ARG;
  }
  // with no rows only dgamma/dbeta are written (zeros, or left as they are
  // when accumulating); the rest may be NULL
  const bool empty = row_count == 0;
  if (!dgamma || (ln && !dbeta)) return SP_ERR_INVALID_ARG;
  if (!empty && (!dy || !h_saved || !gamma || !rstd || !d_residual || !d_sum))
    return SP_ERR_INVALID_ARG;
  if (!empty && ln && !mean) return SP_ERR_INVALID_ARG;
  if (!empty) {  // the range's first row of every per-row argument
    const int64_t rowb = pr.H * elem_bytes(pr.dtype);
    dy = static_cast<const char*>(dy) + row_begin * rowb;
    if (dh_out) dh_out = static_cast<const char*>(dh_out) + row_begin * rowb;
    h_saved = static_cast<const char*>(h_saved) + row_begin * rowb;
    if (mask) mask += row_begin * pr.H;
    rstd += row_begin;
    if (ln) mean += row_begin;
    d_residual = static_cast<char*>(d_residual) + row_begin * rowb;
    d_sum = static_cast<char*>(d_sum) + row_begin * rowb;
  }
  if (!aligned(dy, 16) || (dh_out && !aligned(dh_out, 16)) || !aligned(h_saved, 16) ||
      !aligned(gamma, 16) || (mask && !aligned(mask, 16)) || !aligned(rstd, 4) ||
      (ln && !aligned(mean, 4)) || !aligned(d_residual, 16) || !aligned(d_sum, 16) ||
      !aligned(dgamma, 16) || (ln && !aligned(dbeta, 16)))
    return SP_ERR_ALIGN;
  if (empty && accumulate) return SP_OK;  // nothing to add, nothing launched
  Problem prr = pr;  // the rows this call processes
  prr.rows = row_count;
  BwdPlan pl;
  st = plan_bwd(prr, dh_out != nullptr, desc->p > 0.0f && mask != nullptr, &pl);
  if (st != SP_OK) return st;
  if (!workspace || workspace_bytes < pl.ws_bytes) return SP_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return SP_ERR_ALIGN;
  if (inject_launch_failure()) return SP_ERR_CUDA;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  int nparts = 0;
  if (!empty) {
    BwdArgs a = {};
    a.dy = dy;
    a.dh = dh_out;
    a.h = h_saved;
    a.gamma = gamma;
    a.mask = desc->p > 0.0f ? mask : nullptr;
    a.regen = desc->p > 0.0f && !mask ? 1 : 0;
    a.thr = (uint32_t)std::floor((double)desc->p * 4294967296.0);
    a.grow0 = (int64_t)pr.j * pr.R + row_begin;
    for (int i = 0; i < 10; ++i) {
      a.keys.rk[2 * i] = (uint32_t)desc->seed + (uint32_t)i * 0x9E3779B9u;
      a.keys.rk[2 * i + 1] = (uint32_t)(desc->seed >> 32) + (uint32_t)i * 0xBB67AE85u;
    }
    a.rstd = rstd;
    a.mean = ln ? mean : nullptr;
    a.d_res = d_residual;
    a.d_sum = d_sum;
    a.ws = ws;
    a.rows = row_count;
    a.rows_per_cta = pl.rows_per_cta;
    a.H = (int32_t)pr.H;
    a.nvec = pr.nvec;
    a.tpr = pl.shape.tpr;
    a.nparts = pl.nparts;
    a.scale = (float)(1.0 / (1.0 - (double)desc->p));
    a.Hf = (float)pr.H;
    a.status = desc->status;
    a.wait_ns = wait_hooks().wait_ns;
    a.drop_stage = wait_hooks().drop_stage;
    cudaError_t e;
    if (pl.tma) {
      a.tpr = pl.tp.shape.tpr;
      e = launch_bwd_tma(ln, a, pl.tp, dim3((unsigned)pl.ctas), cs);
    } else {
      e = launch_bwd(pr.dtype, ln, a, pl.shape, dim3((unsigned)pl.ctas), pl.smem, cs);
    }
    if (e != cudaSuccess) return from_cuda(e);
    nparts = pl.nparts;
  }
  return from_cuda(launch_colsum(ws, nparts, (int)pr.H, ln, dgamma, ln ? dbeta : nullptr, accumulate, cs));
}


}  // namespace
}  // namespace spf

using namespace spf;

extern "C" {

sp_status_t sp_rs_dropout_residual_norm_fwd(const sp_rs_desc_t* desc, const void* const* partials,
                                            const void* residual, const void* gamma,
                                            const void* beta, void* h_out, void* y_out,
                                            uint8_t* mask_out, float* rstd_out, float* mean_out,
                                            sp_stream_t stream) {
  return fwd_impl(desc, false, 0, 0, partials, residual, gamma, beta, h_out, y_out, mask_out, rstd_out,
                  mean_out, stream);
}

sp_status_t sp_rs_dropout_residual_norm_fwd_rows(const sp_rs_desc_t* desc, int64_t row_begin,
                                                 int64_t row_count, const void* const* partials,
                                                 const void* residual, const void* gamma,
                                                 const void* beta, void* h_out, void* y_out,
                                                 uint8_t* mask_out, float* rstd_out, float* mean_out,
                                                 sp_stream_t stream) {
  return fwd_impl(desc, true, row_begin, row_count, partials, residual, gamma, beta, h_out, y_out,
                  mask_out, rstd_out, mean_out, stream);
}

size_t sp_rs_bwd_workspace_bytes(const sp_rs_desc_t* desc) {
  Problem pr;
  if (check_desc(desc, &pr) != SP_OK) return 0;
  BwdPlan pl;
  if (plan_bwd(pr, true, true, &pl) != SP_OK) return 0;
  return pl.ws_bytes;
}

sp_status_t sp_rs_dropout_residual_norm_bwd(const sp_rs_desc_t* desc, const void* dy,
                                            const void* dh_out, const void* h_saved,
                                            const void* gamma, const uint8_t* mask,
                                            const float* rstd, const float* mean,
                                            void* d_residual, void* d_sum, float* dgamma,
                                            float* dbeta, void* workspace, size_t workspace_bytes,
                                            sp_stream_t stream) {
  return bwd_impl(desc, false, 0, 0, false, dy, dh_out, h_saved, gamma, mask, rstd, mean, d_residual,
                  d_sum, dgamma, dbeta, workspace, workspace_bytes, stream);
}

sp_status_t sp_rs_dropout_residual_norm_bwd_rows(const sp_rs_desc_t* desc, int64_t row_begin,
                                                 int64_t row_count, int32_t accumulate,
                                                 const void* dy, const void* dh_out,
                                                 const void* h_saved, const void* gamma,
                                                 const uint8_t* mask, const float* rstd,
                                                 const float* mean, void* d_residual, void* d_sum,
                                                 float* dgamma, float* dbeta, void* workspace,
                                                 size_t workspace_bytes, sp_stream_t stream) {
  return bwd_impl(desc, true, row_begin, row_count, accumulate != 0, dy, dh_out, h_saved, gamma, mask,
                  rstd, mean, d_residual, d_sum, dgamma, dbeta, workspace, workspace_bytes, stream);
}

static sp_status_t layout_call(bool to_hp, const void* in, void* out, int64_t N, int64_t H,
                               int32_t T, int32_t dtype, sp_stream_t stream) {
  if (dtype != SP_F32 && dtype != SP_BF16) return SP_ERR_DTYPE;
  if (!in || !out) return SP_ERR_INVALID_ARG;
  if (T < 1 || T > kMaxT) return SP_ERR_INVALID_ARG;
  if (N < 0 || H <= 0 || N % T != 0 || H % T != 0) return SP_ERR_SHAPE;
  const int ev = 16 / elem_bytes(dtype);
  if ((H / T) % ev != 0) return SP_ERR_SHAPE;
  if (N > 0 && N > ((int64_t)1 << 50) / H) return SP_ERR_SHAPE;
  if (!aligned(in, 16) || !aligned(out, 16)) return SP_ERR_ALIGN;
  if (inject_launch_failure()) return SP_ERR_CUDA;
  return from_cuda(launch_layout(to_hp, in, out, N, H, T, elem_bytes(dtype),
                                 reinterpret_cast<cudaStream_t>(stream)));
}

sp_status_t sp2hp(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t dtype,
                  sp_stream_t stream) {
  return layout_call(true, in, out, N, H, T, dtype, stream);
}

sp_status_t hp2sp(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t dtype,
                  sp_stream_t stream) {
  return layout_call(false, in, out, N, H, T, dtype, stream);
}

const char* sp_status_string(sp_status_t s) {
  switch (s) {
    case SP_OK: return "SP_OK";
    case SP_ERR_INVALID_ARG: return "SP_ERR_INVALID_ARG: invalid argument";
    case SP_ERR_SHAPE: return "SP_ERR_SHAPE: unsupported or inconsistent shape";
    case SP_ERR_ALIGN: return "SP_ERR_ALIGN: pointer not aligned as required";
    case SP_ERR_DTYPE: return "SP_ERR_DTYPE: unknown dtype or norm";
    case SP_ERR_WORKSPACE: return "SP_ERR_WORKSPACE: workspace missing or too small";
    case SP_ERR_CUDA: return "SP_ERR_CUDA: CUDA runtime error";
    case SP_ERR_NOT_IMPLEMENTED: return "SP_ERR_NOT_IMPLEMENTED";
    default: return "unknown sp_status_t";
  }
}

int32_t sp_version(void) { return 300; }

#ifndef SPF_SOURCE_HASH
#define SPF_SOURCE_HASH "unknown"
#endif
const char* sp_build_hash(void) { return SPF_SOURCE_HASH; }

sp_status_t sp_plan_describe(const sp_rs_desc_t* desc, int32_t sms, int32_t smem_optin,
                             int32_t has_dh, int32_t has_mask, sp_plan_info_t* out) {
  Problem pr;
  sp_status_t st = check_desc(desc, &pr);
  if (st != SP_OK) return st;
  if (!out || sms < 1 || smem_optin < 1) return SP_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  if (pr.dtype != SP_BF16) return SP_OK;  // f32 runs the register-resident kernels
  const bool ln = pr.norm == SP_LAYERNORM;
  FwdTmaPlan tp;
  // the forward launches nothing without rows
  if (pr.rows > 0 && plan_fwd_tma(pr.H, pr.T, ln, smem_optin, pr.rows, sms, &tp)) {
    sp_kernel_plan_t& f = out->fwd;
    f.tma = 1;
    f.block = tp.shape.block;
    f.nthr = tp.nthr;
    f.tpr = tp.shape.tpr;
    f.vpt = tp.shape.vpt;
    f.row_groups = tp.layout.nrg;
    f.rows_per_stage = tp.layout.rb;
    f.stages = tp.layout.nst;
    f.chunked = tp.chunked ? 1 : 0;
    f.stage_bytes = tp.layout.stage_bytes;
    f.smem_bytes = (int64_t)tp.smem;
    f.rows_per_cta = tp.layout.rows_per_cta;
    f.ctas = (pr.rows + tp.layout.rows_per_cta - 1) / tp.layout.rows_per_cta;
  }
  BwdPlan bp;
  // as the backward itself: the mask is read only when p > 0
  if (plan_bwd_tma_for(pr, has_dh != 0, has_mask != 0 && desc->p > 0.0f, sms, smem_optin, &bp)) {
    sp_kernel_plan_t& b = out->bwd;
    b.tma = 1;
    b.block = bp.tp.shape.block;
    b.nthr = bp.tp.nthr;
    b.tpr = bp.tp.shape.tpr;
    b.vpt = bp.tp.shape.vpt;
    b.row_groups = bp.tp.layout.nrg;
    b.rows_per_stage = bp.tp.layout.rb;
    b.stages = bp.tp.layout.nst;
    b.stage_bytes = bp.tp.layout.stage_bytes;
    b.smem_bytes = (int64_t)bp.tp.smem;
    b.rows_per_cta = bp.rows_per_cta;
    b.ctas = bp.ctas;
    b.workspace_bytes = (int64_t)bp.ws_bytes;
    b.noalloc_fits = noalloc_scratch_fits(bp.ws_bytes) ? 1 : 0;
  }
  return SP_OK;
}

const char* sp_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

}  // extern "C"
