// spec_verify_accept_noalloc: spec_verify_accept with its scratch in a static device array, for
// callers that cannot allocate device memory (see include/spectree.h for the contract).

#include <mutex>

#include <cuda_runtime.h>

#include "spectree.h"

namespace {

// Scratch of the no-allocation entry point.  Device memory reserved for as long as the library
// is loaded; host code must not use this name as an address (it is a host-side stand-in), only
// the pointer that cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" spec_status spec_verify_accept_noalloc(const spec_verify_args* args, int32_t* dev_status,
                                                  void* stream) {
  const size_t need = spec_verify_accept_workspace(args);
  if (need == 0) return spec_verify_accept(args, nullptr, 0, dev_status, stream);  // argument error
  if (need > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SPEC_ERR_CUDA;
  return spec_verify_accept(args, scratch, SPEC_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
