// flce_static_scratch.cu - a forward entry point that allocates nothing and needs no workspace.
//
// Some callers cannot hand the library a device workspace: a plain C or foreign-language host
// program with no device allocator of its own, or a service whose device-memory budget is
// fixed when it starts and which may not call cudaMalloc while it runs (cudaMalloc can also
// synchronise the device). For them, flce_forward_static_scratch() runs the same forward as
// flce_forward() with its scratch placed in one file-scope device array of fixed size.
//
// Costs and limits:
//   * The array (FLCE_STATIC_SCRATCH_BYTES, 64 MiB) is device memory of this file's module. It
//     is reserved in a CUDA context when the module is loaded there: with CUDA's default lazy
//     module loading that is the first call of this entry point in the context (the first
//     lookup below), and it stays reserved until the context is destroyed or the process
//     exits. A caller with a fixed memory budget should make one small call at start-up, so
//     that the reservation (which can fail for lack of memory, as FLCE_ERR_CUDA) happens then.
//   * A problem whose forward scratch (flce_forward_workspace_size) exceeds the array is
//     rejected with FLCE_ERR_WORKSPACE before anything is enqueued. bf16 problems up to about
//     T = 16700 tokens fit at V = 128256; fp32 problems also keep their TF32 hi/lo copies of x
//     and weight there, 8 (T + V) H bytes, so only small ones fit.
//   * All calls in a context share the one array. Its contents survive from call to call; the
//     forward overwrites every scratch value it later reads, and its tile counter is reset by
//     a memset enqueued with each call, so nothing has to start at zero. Two calls whose GPU
//     work overlaps (e.g. on two streams without ordering) race on it.
//   * The array's host-side name is only a stand-in for the symbol, never a device address.
//     The device address is looked up with cudaGetSymbolAddress, with the caller's context
//     current, once per CUDA context (a context has its own copy of the array, and a device's
//     primary context that is reset and created again may place it elsewhere), and cached
//     under the context's unique id. That first call in a context should come before any
//     stream capture.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "flce_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(FLCE_STATIC_SCRATCH_BYTES);

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Driver entry points for the current context and its process-unique id (looked up once).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return fns;
}

// Id of the context current on this thread, or 0 when there is none or it cannot be read.
unsigned long long current_context_id() {
  const DriverFns& f = driver_fns();
  if (!f.get_current || !f.get_id) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// (context id, device address of g_static_scratch in that context). Ids are never reused
// within a process, so an entry can never be mistaken for another context's.
constexpr int kCacheEntries = 64;
struct CacheEntry {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_scratch_mu;
CacheEntry g_cache[kCacheEntries] = {};
int g_cache_used = 0;

// Device address of g_static_scratch in the caller's current context. The lookup itself always
// resolves the symbol in the current context; the cache only skips repeating it.
int static_scratch_address(void** out) {
  unsigned long long id = current_context_id();
  if (id != 0) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    for (int i = 0; i < g_cache_used; ++i) {
      if (g_cache[i].ctx_id == id) {
        *out = g_cache[i].addr;
        return FLCE_OK;
      }
    }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
    return FLCE_ERR_CUDA;
  // With no context current before, the lookup created (and made current) the device's
  // primary context: read its id now.
  if (id == 0) id = current_context_id();
  if (id != 0) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    bool known = false;
    for (int i = 0; i < g_cache_used && !known; ++i) known = g_cache[i].ctx_id == id;
    // beyond kCacheEntries contexts (or without an id) the lookup is repeated on every call
    if (!known && g_cache_used < kCacheEntries) g_cache[g_cache_used++] = CacheEntry{id, p};
  }
  *out = p;
  return FLCE_OK;
}

}  // namespace

extern "C" int flce_forward_static_scratch(const void* x, const void* weight,
                                           const int64_t* target, int64_t T, int64_t H,
                                           int64_t V, int dtype, int reduction, float* loss,
                                           float* lse, int* status, void* stream) {
  if (!x || !weight || !target || !loss || !lse || !status) return FLCE_ERR_ARG;
  const size_t need = flce_forward_workspace_size(T, H, V, dtype);
  if (need == 0) return FLCE_ERR_ARG;
  if (need > kStaticScratchBytes) return FLCE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = static_scratch_address(&scratch);
  if (rc != FLCE_OK) return rc;
  return flce_forward(x, weight, target, T, H, V, dtype, reduction, loss, lse, scratch,
                      kStaticScratchBytes, status, stream);
}
