// flce_static_scratch.cu - a forward entry point that allocates nothing and needs no workspace.
//
// Some callers cannot hand the library a device workspace: a plain C or foreign-language host
// program with no device allocator of its own, or a service whose device-memory budget is
// fixed when it starts and which may not call cudaMalloc while it runs (cudaMalloc can also
// synchronise the device). For them, flce_forward_static_scratch() runs the same forward as
// flce_forward() with its scratch placed in one file-scope device array of fixed size.
//
// Costs and limits:
//   * Every GPU that loads this library holds FLCE_STATIC_SCRATCH_BYTES (64 MiB) for this
//     array until the process exits, whether or not the entry point is ever called.
//   * A problem whose forward scratch (flce_forward_workspace_size) exceeds the array is
//     rejected with FLCE_ERR_WORKSPACE before anything is enqueued.
//   * All calls on a device share the one array. Its contents survive from call to call; the
//     forward overwrites every scratch value it later reads, so nothing has to start at zero.
//     Two calls whose GPU work overlaps (e.g. on two streams without ordering) race on it.
//   * The array's host-side name is only a stand-in for the symbol, never a device address:
//     the device address is looked up once per device with cudaGetSymbolAddress, on the first
//     call made while that device is current. That first call on each device should therefore
//     come before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "flce_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(FLCE_STATIC_SCRATCH_BYTES);

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once per device).
int static_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return FLCE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" int flce_forward_static_scratch(const void* x, const void* weight,
                                           const int64_t* target, int64_t T, int64_t H,
                                           int64_t V, int dtype, int reduction, float* loss,
                                           float* lse, int* status, void* stream) {
  const size_t need = flce_forward_workspace_size(T, H, V, dtype);
  if (need == 0) return FLCE_ERR_ARG;
  if (need > kStaticScratchBytes) return FLCE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = static_scratch_address(&scratch);
  if (rc != FLCE_OK) return rc;
  return flce_forward(x, weight, target, T, H, V, dtype, reduction, loss, lse, scratch,
                      kStaticScratchBytes, status, stream);
}
