// mha_no_alloc.cu - mha_forward_no_alloc: the whole forward pass with its
// intermediates (head-split Q, K, V, the concatenated Z and the device error
// word) kept in a fixed array of device memory that is part of this library,
// so the call itself allocates nothing.
//
// Some callers cannot call cudaMalloc or hand over a workspace: code running
// where device allocation is forbidden or unavailable (inside a host
// framework that owns every device allocation, a plugin with a fixed memory
// budget, a real-time loop that must not allocate after start-up). They pass
// only their inputs and outputs.
#include <mutex>

#include "internal.h"

namespace {

// The scratch: MHA_NO_ALLOC_SCRATCH_BYTES of device memory. Every GPU on
// which this library's device code is loaded holds it until the process exits.
static __device__ __align__(256) unsigned char g_scratch[MHA_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_scratch on the current device. In host code the name
// g_scratch is only a host-side stand-in, so the address is asked of the
// runtime once per device (the first call on that device) and cached.
mha_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MHA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MHA_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return MHA_OK;
}

}  // namespace

extern "C" mha_status mha_forward_no_alloc(const void* X_q, const void* X_kv, const void* W_Q,
                                           const void* W_K, const void* W_V, const void* W_O,
                                           void* Y, int B, int n_q, int n_k, int d_model, int h,
                                           int d_h, int d_vh, int d_o, float c,
                                           mha_mask_kind mask, const int32_t* valid_len,
                                           mha_dtype dt, void* stream) {
  // Sizes beyond the fixed scratch are rejected before any CUDA call.
  const size_t need = mha_workspace_size(B, n_q, n_k, d_model, h, d_h, d_vh, d_o, dt);
  if (need == 0) return MHA_ERR_INVALID_ARG;
  if (need > (size_t)MHA_NO_ALLOC_SCRATCH_BYTES) return MHA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const mha_status st = scratch_address(&scratch);
  if (st != MHA_OK) return st;
  // The same checks and kernels as mha_forward, on the fixed scratch; it also
  // resets the error word (the first 4 bytes) before the kernels run.
  return mha_forward(X_q, X_kv, W_Q, W_K, W_V, W_O, Y, B, n_q, n_k, d_model, h, d_h, d_vh, d_o,
                     c, mask, valid_len, dt, scratch, (size_t)MHA_NO_ALLOC_SCRATCH_BYTES, stream);
}
