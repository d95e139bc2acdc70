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

// Device address of the scratch array on the current device.  Outside a stream capture the
// address is looked up on every call (so a device reset that moved the array is followed) and
// remembered; during a capture, runtime queries that are not stream work are avoided and the
// remembered address is used.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  err = cudaStreamIsCapturing(stream, &cap);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  } else if (!g_scratch_ptr[dev]) {
    return cudaErrorStreamCaptureUnsupported;  // no call on this device before the capture
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
  if (scratch_address(static_cast<cudaStream_t>(stream), &scratch) != cudaSuccess) return SPEC_ERR_CUDA;
  return spec_verify_accept(args, scratch, SPEC_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
