// wtconv_bwd_weight_noalloc: the parameter-gradient call for callers that
// cannot allocate device memory.
//
// wtconv_bwd_weight needs a caller-provided workspace for its per-CTA
// partial sums.  Some callers have no way to obtain one: a plugin running
// inside a host application that owns the whole device-memory budget (a
// fixed arena or an allocator the plugin cannot reach), or a latency-bound
// caller that must not call cudaMalloc because it can synchronise the
// device.  For them this entry point uses a fixed scratch array that lives
// in the library itself (a static __device__ array, allocated when the
// library's device code is loaded on a GPU and held until the process
// exits), so it allocates nothing.  The method's paper has no counterpart
// of this; it is a packaging convenience.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/wtconv.h"
#include "wtconv_launch.h"

namespace {

// 4 MiB: enough for every WTConvNeXt-T layer shape (the largest partial-sum
// record set there is about 1.7 MB).
constexpr size_t kScratchBytes = 4u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_scratch[kScratchBytes / sizeof(float)];

std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  In host code
// `g_scratch` names a host-side shadow, not device memory, so it must never be
// passed to a kernel directly.  Outside stream capture the address is looked
// up on every call (a cudaDeviceReset reloads the device code, which may move
// the array) and kept per device; inside a capture, where the lookup could
// load code, the kept address from an earlier call is used.
wtconv_status_t scratch_for_current_device(cudaStream_t stream, float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "wtconv_bwd_weight_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
    wt::set_last_error(msg);
    return WTCONV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    wt::set_last_error("wtconv_bwd_weight_noalloc: device ordinal beyond the supported 64 devices");
    return WTCONV_ERR_UNSUPPORTED;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "wtconv_bwd_weight_noalloc: cudaStreamIsCapturing failed: %s",
             cudaGetErrorString(e));
    wt::set_last_error(msg);
    return WTCONV_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof(msg), "wtconv_bwd_weight_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      wt::set_last_error(msg);
      return WTCONV_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  } else if (g_scratch_ptr[dev] == nullptr) {
    wt::set_last_error("wtconv_bwd_weight_noalloc: the first call on a device must come before any stream "
                       "capture (it looks up the scratch array's device address)");
    return WTCONV_ERR_INVALID_ARG;
  }
  *out = g_scratch_ptr[dev];
  return WTCONV_OK;
}

}  // namespace

extern "C" wtconv_status_t wtconv_bwd_weight_noalloc(
    const wtconv_desc_t* desc, const void* x, const void* dy, const float* w_base, const float* b_base,
    const float* w_sub, const float* base_scale, const float* wavelet_scale, float* dw_base,
    float* db_base, float* dw_sub, float* dbase_scale, float* dwavelet_scale, void* stream) {
  const size_t need = wtconv_workspace_size(desc, WTCONV_OP_BWD_WEIGHT);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "wtconv_bwd_weight_noalloc: this layer needs %zu bytes of scratch but the library's "
             "static scratch holds %zu; call wtconv_bwd_weight with a workspace instead",
             need, kScratchBytes);
    wt::set_last_error(msg);
    return WTCONV_ERR_UNSUPPORTED;
  }
  if (need == 0) {
    // Invalid descriptor, empty batch or unsupported plane: the regular call
    // reports it (or, for an empty batch, writes zero gradients) without
    // touching any workspace.
    return wtconv_bwd_weight(desc, x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, dw_base, db_base,
                             dw_sub, dbase_scale, dwavelet_scale, nullptr, 0, stream);
  }
  float* scratch = nullptr;
  const wtconv_status_t st = scratch_for_current_device(static_cast<cudaStream_t>(stream), &scratch);
  if (st != WTCONV_OK) return st;
  // Every partial-sum record is written before it is read, so the stale
  // contents left by an earlier call need no clearing.
  return wtconv_bwd_weight(desc, x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, dw_base, db_base,
                           dw_sub, dbase_scale, dwavelet_scale, scratch, kScratchBytes, stream);
}
