// Forward pass without a caller-provided workspace, for callers that cannot allocate device
// memory: code running inside a CUDA graph being captured by someone else, host code bound to
// a fixed memory budget or a custom allocator it may not bypass, or plugins that only receive
// input and output pointers.  The workspace comes from one file-scope device array of
// kStaticWorkspaceBytes; this entry point allocates nothing and calls no allocating routine.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace upipe {
upipe_status_t cuda_status(cudaError_t e);
}

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;  // 32 MiB, held by every GPU that loads the library
constexpr int kMaxDevices = 64;

// The workspace itself.  In host code this name is only a stand-in for the device symbol:
// its device address is obtained with cudaGetSymbolAddress below and passed to the kernels.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {};

// Device address of the array on the current device, resolved once per device (no allocation).
upipe_status_t static_workspace(void** ws) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return upipe::cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return UPIPE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_device_ptr[dev]) {
    // first call on this device: the device is current, so the symbol resolves to its copy
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess) return upipe::cuda_status(e);
    g_device_ptr[dev] = p;
  }
  *ws = g_device_ptr[dev];
  return UPIPE_OK;
}

}  // namespace

extern "C" upipe_status_t upipe_attn_fwd_no_alloc(const upipe_attn_desc_t* desc, const uint16_t* X,
                                                  const uint16_t* Wqkv, const uint16_t* Wo, const int32_t* seg,
                                                  uint16_t* Y, float* lse, void* stream) {
  size_t need = 0;
  upipe_status_t s = upipe_attn_workspace_size(desc, 0, &need);
  if (s != UPIPE_OK) return s;
  if (need > kStaticWorkspaceBytes) return UPIPE_ERR_WORKSPACE_TOO_SMALL;  // descriptor too large for the array
  void* ws = nullptr;
  s = static_workspace(&ws);
  if (s != UPIPE_OK) return s;
  // every buffer that must start from a known state (the table header with its error word, the
  // first chunk's output accumulator) is initialised by the forward pass itself
  return upipe_attn_fwd(desc, X, Wqkv, Wo, seg, Y, lse, ws, kStaticWorkspaceBytes, stream);
}

// The array's error word (the table header at its base), read like any workspace's.  Before the
// first forward on a device the array is still zero-initialised, so the word reads UPIPE_OK.
extern "C" upipe_status_t upipe_attn_no_alloc_device_status(int32_t* code, void* stream) {
  if (!code) return UPIPE_ERR_INVALID_ARG;
  void* ws = nullptr;
  upipe_status_t s = static_workspace(&ws);
  if (s != UPIPE_OK) return s;
  return upipe_attn_device_status(ws, code, stream);
}
