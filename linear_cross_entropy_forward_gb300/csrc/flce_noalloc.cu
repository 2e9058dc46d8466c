// flce_forward_noalloc: the forward pass for callers that cannot allocate device
// memory.  It has no counterpart in the pages; it exists because some callers can't
// call cudaMalloc: a framework or serving runtime may hand out all device memory up
// front and keep it, or the caller may run under an allocator it does not own, and
// then there is no way to provide the workspace flce_forward needs.
//
// Instead of a caller-supplied workspace it uses the file-scope device array
// below, FLCE_NOALLOC_SCRATCH_BYTES (64 MiB) per GPU.  Every GPU that loads this
// library keeps that array until the process exits.  Host code never touches
// the array by name: at set-up, once per device and with that device current,
// the device address is fetched with cudaGetSymbolAddress and handed to the
// regular forward launch sequence as its workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/flce.h"

namespace {

constexpr size_t kScratchBytes = FLCE_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_flce_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_flce_scratch on the current device (set-up on first use).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_flce_scratch) != cudaSuccess || !p) return FLCE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" int flce_forward_noalloc(const flce_params* params, const void* hidden,
                                    const void* weight, const int64_t* labels, float* loss,
                                    float* entropy, float* lse, float* ez, void* stream) {
  const size_t need = flce_workspace_size(params, 0);
  // invalid parameters: let the regular argument checks report the exact code
  if (need == 0)
    return flce_forward(params, hidden, weight, labels, loss, entropy, lse, ez, nullptr, 0,
                        stream);
  if (need > kScratchBytes) return FLCE_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != FLCE_OK) return rc;
  return flce_forward(params, hidden, weight, labels, loss, entropy, lse, ez, scratch,
                      kScratchBytes, stream);
}
