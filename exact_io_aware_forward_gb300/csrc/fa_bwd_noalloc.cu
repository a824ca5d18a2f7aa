// fa_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// fa_backward needs a caller-provided workspace (the D vector and the fp32 dQ
// accumulator).  Some callers have no way to get one: code running inside a
// host framework that owns every device allocation and exposes no allocator
// to plugins, allocation-free real-time / inference paths that must not call
// cudaMalloc after start-up, and callers that only receive raw device
// pointers for their inputs and outputs.  This entry point uses instead a
// fixed scratch array that lives in the library's own device image.
//
// Cost and limits:
//   * Every GPU that loads the library holds FA_NOALLOC_SCRATCH_BYTES of
//     device memory for this array until the process exits.
//   * Problems whose workspace (fa_backward_workspace_size) exceeds that size
//     are rejected with FA_ERR_SCRATCH_TOO_SMALL before anything is launched.
//   * The first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture begins.
//   * All calls on one device share the one array.  Calls whose work
//     overlaps on the GPU (different streams, no ordering between them) race
//     on it and give wrong gradients; serialise them.
//   * The array keeps the previous call's contents; the preprocess stage
//     rewrites D and clears the dQ accumulator to zero on every call.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = FA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                                         const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                                         int H, int N, int d, int dtype, int causal, float scale,
                                         void* stream) {
  // Invalid arguments get the status fa_backward gives them, before any CUDA
  // call; only then does the size of the problem matter.
  const int st = fa::backward_arguments_status(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, dtype, scale);
  if (st != FA_OK) return static_cast<fa_status>(st);
  if (fa_backward_workspace_size(B, H, N, d) > kScratchBytes) return FA_ERR_SCRATCH_TOO_SMALL;
  void* base = scratch_on_current_device();
  if (base == nullptr) return FA_ERR_CUDA;
  // D and the dQ accumulator are laid out in the scratch exactly as in a
  // caller's workspace.
  return fa_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, dtype, causal, scale, base, kScratchBytes,
                     stream);
}
