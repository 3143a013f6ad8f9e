// noalloc.cu -- backward entry point that needs no caller-provided workspace.
//
// The dgamma/dbeta partial rows live in a fixed device array declared in this
// file, so the call allocates nothing.  The array is reserved on every GPU
// that loads the library and stays reserved until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/spfuse.h"
#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;

// Backing store of the scratch; its size is SP_NOALLOC_SCRATCH_BYTES.
static __device__ __align__(256) unsigned char g_bwd_scratch[SP_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device.  On the host the
// symbol g_bwd_scratch is only a stand-in, so the address is asked of the
// runtime once per device, with that device current, and cached.
sp_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return SP_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SP_OK;
}

}  // namespace

extern "C" sp_status_t sp_rs_dropout_residual_norm_bwd_noalloc(
    const sp_rs_desc_t* desc, const void* dy, const void* dh_out, const void* h_saved,
    const void* gamma, const uint8_t* mask, const float* rstd, const float* mean,
    void* d_residual, void* d_sum, float* dgamma, float* dbeta, sp_stream_t stream) {
  // A problem whose partial rows need more than the fixed array is refused
  // before anything is launched (an invalid descriptor reports 0 here and is
  // refused with its own status by the call below).
  if (!spf::noalloc_scratch_fits(sp_rs_bwd_workspace_bytes(desc))) return SP_ERR_WORKSPACE;
  void* scratch = nullptr;
  const sp_status_t st = scratch_for_current_device(&scratch);
  if (st != SP_OK) return st;
  // Same validation and kernels as the workspace entry point.
  return sp_rs_dropout_residual_norm_bwd(desc, dy, dh_out, h_saved, gamma, mask, rstd, mean,
                                         d_residual, d_sum, dgamma, dbeta, scratch,
                                         (size_t)SP_NOALLOC_SCRATCH_BYTES, stream);
}
