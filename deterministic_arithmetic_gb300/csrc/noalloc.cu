// noalloc.cu -- a forward pass for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// under an allocator it does not own (a framework's caching allocator that
// must not be bypassed, an inference server that pre-plans every byte), or a
// host program without a CUDA allocator of its own at the call site. For them
// lora_delta_fwd_noalloc runs the same forward kernels as lora_delta_fwd, with
// the scratch (the status block and the FP32 partial sums of U) taken from a
// fixed array that lives in the library's device image instead of from a
// caller-provided workspace.
//
// The array is a file-scope __device__ variable. Host code cannot use its
// name as a device address (on the host the name only stands in for the
// symbol), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current, and every later call on
// that device reuses the address.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/lora_delta.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB, held by every device that loads the library
constexpr size_t kStatusBytes = 256;                 // must be zero when a call starts
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
lora_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return LORA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LORA_OK;
}

// The address if a call on the current device has looked it up already, else null.
void* known_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" lora_status lora_delta_fwd_noalloc(const void* x, const void* a, const void* b, float alpha, int64_t M,
                                              int64_t K, int64_t N, int64_t R, float* delta_y, void* u,
                                              void* stream) {
  const size_t need = lora_delta_fwd_workspace_size(M, K, N, R);
  if (need == 0 || M == 0)   // invalid shape (reported by the checks of lora_delta_fwd) or nothing to do
    return lora_delta_fwd(x, a, b, alpha, M, K, N, R, delta_y, u, nullptr, 0, stream);
  if (need > kScratchBytes) return LORA_ERR_WORKSPACE;   // shape needs more scratch than the fixed array holds
  void* scratch = nullptr;
  lora_status s = scratch_address(&scratch);
  if (s != LORA_OK) return s;
  // The array keeps whatever the previous call left; only the status block
  // has to start at zero (the partial sums are overwritten before they are read).
  if (cudaMemsetAsync(scratch, 0, kStatusBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LORA_ERR_CUDA;
  return lora_delta_fwd(x, a, b, alpha, M, K, N, R, delta_y, u, scratch, kScratchBytes, stream);
}

// The status block is the first word of the array; before any call on this device there is
// nothing to report (the array starts zeroed, as every __device__ variable does).
extern "C" lora_status lora_delta_fwd_noalloc_status(int* code) {
  if (!code) return LORA_ERR_NULL;
  void* scratch = known_scratch_address();
  if (!scratch) {
    *code = 0;
    return LORA_OK;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return LORA_ERR_CUDA;
  return lora_delta_device_status(scratch, code);
}
