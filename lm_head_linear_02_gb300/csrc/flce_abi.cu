// flce_abi.cu - the C ABI of libflce: argument validation, workspace carve-up, TMA tensor-map
// encoding and launch sequencing. All compute runs in the kernels of flce_fwd.cu / flce_bwd.cu;
// this file only checks, plans and enqueues. Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "flce_internal.h"

namespace flce {

// ------------------------------------------------------------------------------- device

bool current_device(Device* d) {
  static std::mutex mu;
  static Device cache[64];
  int id = -1;
  if (cudaGetDevice(&id) != cudaSuccess || id < 0) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (id < 64 && cache[id].id == id) {
    *d = cache[id];
    return true;
  }
  Device x;
  x.id = id;
  if (cudaDeviceGetAttribute(&x.sms, cudaDevAttrMultiProcessorCount, id) != cudaSuccess ||
      cudaDeviceGetAttribute(&x.cc_major, cudaDevAttrComputeCapabilityMajor, id) != cudaSuccess ||
      cudaDeviceGetAttribute(&x.cc_minor, cudaDevAttrComputeCapabilityMinor, id) != cudaSuccess)
    return false;
  if (id < 64) cache[id] = x;
  *d = x;
  return true;
}

// ------------------------------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t inner,
                  uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (row_bytes & 15u) != 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  std::memset(tm, 0, sizeof(*tm));
  return enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------------- tuning

namespace {
std::atomic<int> g_tune_raster_rows{2048};
std::atomic<int> g_tune_raster_vocab{kDefaultRasterVocab};
std::atomic<int> g_tune_split_epilogue{kDefaultSplitEpilogue};
std::atomic<int> g_tune_ordered_drain{kDefaultOrderedDrain};
std::atomic<int> g_tune_sm_pairs{-1};
std::atomic<int> g_tune_wide_tiles{-1};
}  // namespace

int tune_raster_rows() { return g_tune_raster_rows.load(); }
int tune_raster_vocab() { return g_tune_raster_vocab.load(); }
int tune_split_epilogue() { return g_tune_split_epilogue.load(); }
int tune_ordered_drain() { return g_tune_ordered_drain.load(); }

namespace {
std::atomic<int> g_withhold_request{0};
}  // namespace

bool take_withhold_request() { return g_withhold_request.exchange(0) != 0; }
int tune_sm_pairs() { return g_tune_sm_pairs.load(); }
int tune_wide_tiles() { return g_tune_wide_tiles.load(); }

// ------------------------------------------------------------------------------- timing
// Optional event brackets around each contraction launch (see flce_timing_enable).

namespace {
struct TimedLaunch {
  int role;
  cudaEvent_t begin, end;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimedLaunch> g_pending;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

// Runs `launch` (returning cudaError_t); brackets it with events when timing is enabled.
template <class F>
cudaError_t timed_launch(int role, cudaStream_t s, F&& launch) {
  bool on;
  {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    on = g_timing_on;
  }
  if (!on) return launch();
  cudaEvent_t b, e;
  {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    b = take_event();
    e = take_event();
  }
  if (!b || !e) return cudaErrorMemoryAllocation;
  cudaError_t r = cudaEventRecord(b, s);
  if (r != cudaSuccess) return r;
  r = launch();
  if (r != cudaSuccess) return r;
  r = cudaEventRecord(e, s);
  if (r != cudaSuccess) return r;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  g_pending.push_back(TimedLaunch{role, b, e});
  return cudaSuccess;
}

}  // namespace flce

// ================================================================================ C ABI

namespace {

using flce::kTileM;
using flce::kTileN;

constexpr int64_t kMaxDim = int64_t(1) << 24;          // T, V bound (tile counts fit in int)
constexpr int64_t kMaxHidden = int64_t(1) << 20;
constexpr size_t kAlign = 256;
// dz slab (all its copies) per slab. Each slab costs one read-modify-write pass over the fp32
// grad_x accumulator; 1 GiB (4 slabs at T = 16384, V = 128256) measured 1.5% faster per step
// than 512 MiB (8 slabs).
constexpr int64_t kSlabBudgetBytes = int64_t(1) << 30;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }
inline size_t align_up(size_t a) { return (a + kAlign - 1) / kAlign * kAlign; }

int elem_bytes(int dtype) { return dtype == FLCE_DTYPE_BF16 ? 2 : 4; }

bool dims_ok(int64_t T, int64_t H, int64_t V, int dtype) {
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_F32) return false;
  if (T <= 0 || H <= 0 || V <= 0) return false;
  if (T > kMaxDim || V > kMaxDim || H > kMaxHidden) return false;
  if (cdiv(T, kTileM) * cdiv(V, kTileN) >= (int64_t(1) << 31)) return false;
  return true;
}

// Sequential carve-up of a workspace into 256-byte aligned regions.
struct Carver {
  size_t off = 0;
  uint8_t* base = nullptr;
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off = align_up(off + bytes);
    return p;
  }
};

struct FwdWs {
  float *part_m, *part_s, *zy, *sx, *block_sums;
  int* counter;                      // tile counter of the projection launch
  float *x_hi, *x_lo, *w_hi, *w_lo;  // f32 path only: x [T][H]; one weight slab [vf][H]
  int64_t vf;                        // f32 path: weight rows per projection launch
};

// fp32 path: weight rows whose TF32 hi/lo copies the forward holds at once (the projection runs
// slab by slab): at most 256 MB of copies, a multiple of 256, slabs of nearly equal width.
constexpr int64_t kFwdSlabBytesF32 = int64_t(1) << 28;

int64_t fwd_slab_width_f32(int64_t H, int64_t V) {
  const int64_t vmax = round_up(V, kTileN);
  int64_t vf = kFwdSlabBytesF32 / (8 * H) / kTileN * kTileN;
  if (vf < kTileN) vf = kTileN;
  if (vf >= vmax) return vmax;
  return round_up(cdiv(V, cdiv(V, vf)), kTileN);
}

size_t carve_fwd(Carver& c, int64_t T, int64_t H, int64_t V, int dtype, FwdWs* w) {
  const int64_t nt = cdiv(V, kTileN);
  FwdWs r{};
  r.part_m = static_cast<float*>(c.take(sizeof(float) * nt * T));
  r.part_s = static_cast<float*>(c.take(sizeof(float) * nt * T));
  r.zy = static_cast<float*>(c.take(sizeof(float) * T));
  r.sx = static_cast<float*>(c.take(sizeof(float) * T));
  r.block_sums = static_cast<float*>(c.take(sizeof(float) * cdiv(T, flce::kLossBlockTokens)));
  r.counter = static_cast<int*>(c.take(sizeof(int)));
  if (dtype == FLCE_DTYPE_F32) {
    r.vf = fwd_slab_width_f32(H, V);
    r.x_hi = static_cast<float*>(c.take(sizeof(float) * T * H));
    r.x_lo = static_cast<float*>(c.take(sizeof(float) * T * H));
    r.w_hi = static_cast<float*>(c.take(sizeof(float) * r.vf * H));
    r.w_lo = static_cast<float*>(c.take(sizeof(float) * r.vf * H));
  }
  if (w) *w = r;
  return c.off;
}

std::atomic<int64_t> g_slab_override{0};

int64_t slab_width(int64_t T, int64_t H, int64_t V, int dtype) {
  const int64_t vmax = round_up(V, kTileN);
  const int64_t forced = g_slab_override.load();
  if (forced > 0) return forced < vmax ? forced : vmax;
  // bf16: one bf16 slab. f32: dz hi/lo slabs in both [T][Vc] and [Vc][T] orientation, and the
  // weight slab's hi/lo copies in both [Vc][H] and [H][Vc] orientation.
  const int64_t per_col = dtype == FLCE_DTYPE_BF16 ? 2 * T : 16 * round_up(T, 4) + 16 * H;
  int64_t vc = kSlabBudgetBytes / per_col / kTileN * kTileN;
  if (vc < kTileN) vc = kTileN;
  if (vc >= vmax) return vmax;
  // As few slabs as the budget allows, of (nearly) equal width: no narrow last slab.
  return round_up(cdiv(V, cdiv(V, vc)), kTileN);
}

struct BwdWs {
  int64_t vc, n_slabs, ldT, ldVc;
  void* dz;       // bf16 [T][vc] or f32 hi [T][vc]
  float* dz_lo;   // [T][vc]
  float* dzt_hi;  // [vc][ldT]
  float* dzt_lo;
  float* acc;     // bf16 path, [T][H] when more than one slab
  float *x_hi, *x_lo, *xt_hi, *xt_lo;  // [T][H], [H][ldT]
  float *w_hi, *w_lo, *wt_hi, *wt_lo;  // one weight slab: [vc][H], [H][ldVc]
  int* counter;                        // tile counter of the dz and gradient launches
};

size_t carve_bwd(Carver& c, int64_t T, int64_t H, int64_t V, int dtype, BwdWs* w) {
  BwdWs r{};
  r.vc = slab_width(T, H, V, dtype);
  r.n_slabs = cdiv(V, r.vc);
  r.ldT = round_up(T, 4);
  r.ldVc = round_up(r.vc, 4);
  if (dtype == FLCE_DTYPE_BF16) {
    r.dz = c.take(size_t(2) * T * r.vc);
    if (r.n_slabs > 1) r.acc = static_cast<float*>(c.take(sizeof(float) * T * H));
  } else {
    r.dz = c.take(sizeof(float) * T * r.vc);
    r.dz_lo = static_cast<float*>(c.take(sizeof(float) * T * r.vc));
    r.dzt_hi = static_cast<float*>(c.take(sizeof(float) * r.vc * r.ldT));
    r.dzt_lo = static_cast<float*>(c.take(sizeof(float) * r.vc * r.ldT));
    r.x_hi = static_cast<float*>(c.take(sizeof(float) * T * H));
    r.x_lo = static_cast<float*>(c.take(sizeof(float) * T * H));
    r.xt_hi = static_cast<float*>(c.take(sizeof(float) * H * r.ldT));
    r.xt_lo = static_cast<float*>(c.take(sizeof(float) * H * r.ldT));
    r.w_hi = static_cast<float*>(c.take(sizeof(float) * r.vc * H));
    r.w_lo = static_cast<float*>(c.take(sizeof(float) * r.vc * H));
    r.wt_hi = static_cast<float*>(c.take(sizeof(float) * H * r.ldVc));
    r.wt_lo = static_cast<float*>(c.take(sizeof(float) * H * r.ldVc));
  }
  r.counter = static_cast<int*>(c.take(sizeof(int)));
  if (w) *w = r;
  return c.off;
}

struct Range {
  uintptr_t lo, hi;
};
inline Range rng(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}
inline bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- single-call forward + backward (token chunks, no logits recompute)

// bf16 chunk logits per chunk (FLCE_TUNE_CHUNK_BYTES). grad_weight is summed over the chunks in
// its own bf16 output (the first chunk writes it, every later one reads, adds and rounds it
// back), so the workspace holds no V x H accumulator and a chunk count n moves (2n - 1) V H 2
// bytes of grad_weight; 1.5 GiB gives 3 chunks at T = 16384, V = 128256 (workspace 1.46 GB,
// below the 4.2 GB of bf16 logits with x, weight and both gradients included).
constexpr int64_t kMinFusedTokens = 512;
std::atomic<int64_t> g_chunk_bytes{flce::kDefaultChunkBytes};

// The chunked single-call schedule applies to bf16 with at least 512 tokens (so a chunk never
// holds all tokens' logits); otherwise flce_forward_backward runs flce_forward + flce_backward.
bool fused_schedule(int64_t T, int dtype) {
  return dtype == FLCE_DTYPE_BF16 && T >= kMinFusedTokens;
}

int64_t fused_chunk_rows(int64_t T, int64_t V) {
  const int64_t ldz = round_up(V, kTileN);
  int64_t c = g_chunk_bytes.load() / (2 * ldz) / 256 * 256;
  const int64_t half = round_up(cdiv(T, 2), 256);
  if (c > half) c = half;
  if (c < 256) c = 256;
  // As few chunks as the limits allow, of (nearly) equal size: no small last chunk.
  return round_up(cdiv(T, cdiv(T, c)), 256);
}

struct FusedWs {
  int64_t rows, ldz, n_chunks;
  __nv_bfloat16* zbuf;
  float *part_m, *part_s, *zy, *sx, *block_sums;
  int* counter;
};

size_t carve_fused(Carver& c, int64_t T, int64_t H, int64_t V, FusedWs* w) {
  FusedWs r{};
  r.rows = fused_chunk_rows(T, V);
  r.ldz = round_up(V, kTileN);
  r.n_chunks = cdiv(T, r.rows);
  const int64_t nt = r.ldz / (kTileN / 2);  // one partial per 128-column half-tile
  r.zbuf = static_cast<__nv_bfloat16*>(c.take(size_t(2) * r.rows * r.ldz));
  r.part_m = static_cast<float*>(c.take(sizeof(float) * nt * r.rows));
  r.part_s = static_cast<float*>(c.take(sizeof(float) * nt * r.rows));
  r.zy = static_cast<float*>(c.take(sizeof(float) * r.rows));
  r.sx = static_cast<float*>(c.take(sizeof(float) * r.rows));
  r.block_sums = static_cast<float*>(c.take(sizeof(float) * cdiv(T, flce::kLossBlockTokens)));
  r.counter = static_cast<int*>(c.take(sizeof(int)));
  if (w) *w = r;
  return c.off;
}

int check_device(flce::Device* dev) {
  if (!flce::current_device(dev)) return FLCE_ERR_CUDA;
  if (dev->cc_major != 10 || dev->cc_minor != 3) return FLCE_ERR_UNSUPPORTED;
  return FLCE_OK;
}

}  // namespace

extern "C" {

int flce_version(void) { return 10000; }

const char* flce_strerror(int code) {
  switch (code) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_ARG: return "invalid argument (null pointer, size out of range or unknown enum)";
    case FLCE_ERR_UNSUPPORTED:
      return "unsupported (misaligned pointer or row stride, or device is not sm_103)";
    case FLCE_ERR_WORKSPACE: return "workspace missing or smaller than the size query requires";
    case FLCE_ERR_ALIAS: return "an output overlaps an input or another output";
    case FLCE_ERR_CUDA: return "a CUDA runtime or driver call failed";
    default: return "unknown error code";
  }
}

size_t flce_forward_workspace_size(int64_t T, int64_t H, int64_t V, int dtype) {
  if (!dims_ok(T, H, V, dtype)) return 0;
  Carver c;
  return carve_fwd(c, T, H, V, dtype, nullptr);
}

size_t flce_backward_workspace_size(int64_t T, int64_t H, int64_t V, int dtype) {
  if (!dims_ok(T, H, V, dtype)) return 0;
  Carver c;
  return carve_bwd(c, T, H, V, dtype, nullptr);
}

size_t flce_forward_backward_workspace_size(int64_t T, int64_t H, int64_t V, int dtype) {
  if (!dims_ok(T, H, V, dtype)) return 0;
  if (!fused_schedule(T, dtype)) {
    const size_t f = flce_forward_workspace_size(T, H, V, dtype);
    const size_t b = flce_backward_workspace_size(T, H, V, dtype);
    return f > b ? f : b;
  }
  Carver c;
  return carve_fused(c, T, H, V, nullptr);
}

int64_t flce_forward_backward_chunk_tokens(int64_t T, int64_t H, int64_t V, int dtype) {
  if (!dims_ok(T, H, V, dtype)) return 0;
  return fused_schedule(T, dtype) ? fused_chunk_rows(T, V) : T;
}

int64_t flce_backward_slab_width(int64_t T, int64_t H, int64_t V, int dtype) {
  if (!dims_ok(T, H, V, dtype)) return 0;
  return slab_width(T, H, V, dtype);
}

int flce_test_withhold_signal(void) {
  flce::g_withhold_request.store(1);
  return FLCE_OK;
}

int flce_timing_enable(int on) {
  std::lock_guard<std::mutex> lock(flce::g_timing_mu);
  flce::g_timing_on = on != 0;
  return FLCE_OK;
}

int flce_timing_read(int64_t counts[FLCE_TIMING_ROLES], double ms[FLCE_TIMING_ROLES]) {
  if (!counts || !ms) return FLCE_ERR_ARG;
  std::vector<flce::TimedLaunch> done;
  {
    std::lock_guard<std::mutex> lock(flce::g_timing_mu);
    done.swap(flce::g_pending);
  }
  for (int r = 0; r < FLCE_TIMING_ROLES; ++r) {
    counts[r] = 0;
    ms[r] = 0.0;
  }
  int rc = FLCE_OK;
  for (const auto& t : done) {
    float el = 0.f;
    if (cudaEventSynchronize(t.end) != cudaSuccess ||
        cudaEventElapsedTime(&el, t.begin, t.end) != cudaSuccess) {
      rc = FLCE_ERR_CUDA;
      continue;
    }
    if (t.role >= 0 && t.role < FLCE_TIMING_ROLES) {
      counts[t.role] += 1;
      ms[t.role] += el;
    }
  }
  std::lock_guard<std::mutex> lock(flce::g_timing_mu);
  for (const auto& t : done) {
    flce::g_event_pool.push_back(t.begin);
    flce::g_event_pool.push_back(t.end);
  }
  return rc;
}

int flce_set_tuning(int key, int64_t value) {
  switch (key) {
    case FLCE_TUNE_RASTER_ROWS:
      if (value < 256 || value > (int64_t(1) << 20) || value % 256 != 0) return FLCE_ERR_ARG;
      flce::g_tune_raster_rows.store(static_cast<int>(value));
      return FLCE_OK;
    case FLCE_TUNE_SM_PAIRS:
      if (value < -1 || value > 7) return FLCE_ERR_ARG;
      flce::g_tune_sm_pairs.store(static_cast<int>(value));
      return FLCE_OK;
    case FLCE_TUNE_RASTER_VOCAB:
      if (value < 0 || value > (int64_t(1) << 24) || value % 256 != 0) return FLCE_ERR_ARG;
      flce::g_tune_raster_vocab.store(static_cast<int>(value));
      return FLCE_OK;
    case FLCE_TUNE_CHUNK_BYTES:
      if (value < 0 || value > (int64_t(1) << 40)) return FLCE_ERR_ARG;
      g_chunk_bytes.store(value == 0 ? flce::kDefaultChunkBytes : value);
      return FLCE_OK;
    case FLCE_TUNE_SPLIT_EPILOGUE:
      if (value < -1 || value > 7) return FLCE_ERR_ARG;
      flce::g_tune_split_epilogue.store(value < 0 ? flce::kDefaultSplitEpilogue
                                                  : static_cast<int>(value));
      return FLCE_OK;
    case FLCE_TUNE_ORDERED_DRAIN:
      if (value < -1 || value > 7) return FLCE_ERR_ARG;
      flce::g_tune_ordered_drain.store(value < 0 ? flce::kDefaultOrderedDrain
                                                 : static_cast<int>(value));
      return FLCE_OK;
    case FLCE_TUNE_WIDE_TILES:
      if (value < -1 || value > 7) return FLCE_ERR_ARG;
      flce::g_tune_wide_tiles.store(static_cast<int>(value));
      return FLCE_OK;
    default:
      return FLCE_ERR_ARG;
  }
}

int flce_get_tuning(int key, int64_t* value) {
  if (!value) return FLCE_ERR_ARG;
  switch (key) {
    case FLCE_TUNE_RASTER_ROWS:
      *value = flce::g_tune_raster_rows.load();
      return FLCE_OK;
    case FLCE_TUNE_RASTER_VOCAB:
      *value = flce::g_tune_raster_vocab.load();
      return FLCE_OK;
    case FLCE_TUNE_SPLIT_EPILOGUE:
      *value = flce::g_tune_split_epilogue.load();
      return FLCE_OK;
    case FLCE_TUNE_CHUNK_BYTES:
      *value = g_chunk_bytes.load();
      return FLCE_OK;
    case FLCE_TUNE_ORDERED_DRAIN:
      *value = flce::g_tune_ordered_drain.load();
      return FLCE_OK;
    case FLCE_TUNE_SM_PAIRS: {
      flce::Device dev;
      if (!flce::current_device(&dev)) return FLCE_ERR_CUDA;
      *value = flce::pair_roles(dev.sms);
      return FLCE_OK;
    }
    case FLCE_TUNE_WIDE_TILES: {
      const int w = flce::tune_wide_tiles();
      *value = w >= 0 ? w : flce::kDefaultWideRoles;
      return FLCE_OK;
    }
    default:
      return FLCE_ERR_ARG;
  }
}

int flce_set_backward_slab_width(int64_t vc) {
  if (vc < 0 || vc % kTileN != 0 || vc > kMaxDim) return FLCE_ERR_ARG;
  g_slab_override.store(vc);
  return FLCE_OK;
}

int flce_forward(const void* x, const void* weight, const int64_t* target, int64_t T, int64_t H,
                 int64_t V, int dtype, int reduction, float* loss, float* lse, void* workspace,
                 size_t workspace_bytes, int* status, void* stream) {
  // ---- host-side validation (no CUDA call before this block passes)
  if (!x || !weight || !target || !loss || !lse || !status) return FLCE_ERR_ARG;
  if (!dims_ok(T, H, V, dtype)) return FLCE_ERR_ARG;
  if (reduction != FLCE_REDUCTION_SUM && reduction != FLCE_REDUCTION_MEAN &&
      reduction != FLCE_REDUCTION_NONE)
    return FLCE_ERR_ARG;
  const int eb = elem_bytes(dtype);
  if ((H * eb) % 16 != 0 || !aligned16(x) || !aligned16(weight)) return FLCE_ERR_UNSUPPORTED;
  const size_t need = flce_forward_workspace_size(T, H, V, dtype);
  if (!workspace || workspace_bytes < need) return FLCE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return FLCE_ERR_UNSUPPORTED;
  const Range in[3] = {rng(x, size_t(T) * H * eb), rng(weight, size_t(V) * H * eb),
                       rng(target, size_t(T) * 8)};
  const size_t loss_bytes = reduction == FLCE_REDUCTION_NONE ? size_t(T) * 4 : 4;
  const Range out[4] = {rng(loss, loss_bytes), rng(lse, size_t(T) * 4), rng(workspace, need),
                        rng(status, sizeof(int))};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(out[i], in[j])) return FLCE_ERR_ALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(out[i], out[j])) return FLCE_ERR_ALIAS;
  }

  flce::Device dev;
  int rc = check_device(&dev);
  if (rc != FLCE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  Carver c;
  c.base = static_cast<uint8_t*>(workspace);
  FwdWs w;
  carve_fwd(c, T, H, V, dtype, &w);

  flce::FwdLaunch p{};
  p.target = target;
  p.part_m = w.part_m;
  p.part_s = w.part_s;
  p.zy = w.zy;
  p.sx = w.sx;
  p.block_sums = w.block_sums;
  p.lse = lse;
  p.loss = loss;
  p.status = status;
  p.tile_counter = w.counter;
  p.T = int(T);
  p.H = int(H);
  p.V = int(V);
  p.reduction = reduction;
  p.sms = dev.sms;
  p.stream = s;

  cudaError_t e;
  if (dtype == FLCE_DTYPE_BF16) {
    CUtensorMap tx, tw;
    const flce::Core core = flce::role_core(dev.sms, FLCE_ROLE_FORWARD);
    if (!flce::make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, H, T, H * 2, 64,
                            flce::core_a_box_rows(core)) ||
        !flce::make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, weight, H, V, H * 2, 64,
                            flce::core_b_box_rows(core)))
      return FLCE_ERR_CUDA;
    e = flce::timed_launch(0, s, [&] { return flce::launch_forward_bf16(tx, tw, p); });
  } else {
    // x split once; the weight split and projected slab by slab (w.vf rows at a time)
    CUtensorMap txh, txl;
    const auto F = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (!flce::make_tmap_2d(&txh, F, w.x_hi, H, T, H * 4, 32, kTileM) ||
        !flce::make_tmap_2d(&txl, F, w.x_lo, H, T, H * 4, 32, kTileM))
      return FLCE_ERR_CUDA;
    e = flce::launch_split_tf32(static_cast<const float*>(x), T, H, H, w.x_hi, w.x_lo, false, s);
    for (int64_t v0 = 0; v0 < V && e == cudaSuccess; v0 += w.vf) {
      const int64_t sw = (V - v0) < w.vf ? (V - v0) : w.vf;
      CUtensorMap twh, twl;
      const uint32_t wbox =
          flce::core_b_box_rows(flce::tf32_core(dev.sms, FLCE_ROLE_FORWARD));
      if (!flce::make_tmap_2d(&twh, F, w.w_hi, H, sw, H * 4, 32, wbox) ||
          !flce::make_tmap_2d(&twl, F, w.w_lo, H, sw, H * 4, 32, wbox))
        return FLCE_ERR_CUDA;
      e = flce::launch_split_tf32(static_cast<const float*>(weight) + size_t(v0) * H, sw, H, H,
                                  w.w_hi, w.w_lo, false, s);
      if (e == cudaSuccess)
        e = flce::timed_launch(0, s, [&] {
          return flce::launch_forward_tf32(txh, twh, txl, twl, p, int(v0), int(sw));
        });
    }
    if (e == cudaSuccess) e = flce::launch_forward_combine(p);
  }
  return e == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}

int flce_backward(const void* x, const void* weight, const int64_t* target, const float* lse,
                  int64_t T, int64_t H, int64_t V, int dtype, int reduction,
                  const float* grad_loss, void* grad_x, void* grad_weight, void* workspace,
                  size_t workspace_bytes, int* status, void* stream) {
  if (!x || !weight || !target || !lse || !grad_loss || !grad_x || !grad_weight || !status)
    return FLCE_ERR_ARG;
  if (!dims_ok(T, H, V, dtype)) return FLCE_ERR_ARG;
  if (reduction != FLCE_REDUCTION_SUM && reduction != FLCE_REDUCTION_MEAN &&
      reduction != FLCE_REDUCTION_NONE)
    return FLCE_ERR_ARG;
  const int eb = elem_bytes(dtype);
  if ((H * eb) % 16 != 0 || !aligned16(x) || !aligned16(weight) || !aligned16(grad_x) ||
      !aligned16(grad_weight))
    return FLCE_ERR_UNSUPPORTED;
  const size_t need = flce_backward_workspace_size(T, H, V, dtype);
  if (!workspace || workspace_bytes < need) return FLCE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return FLCE_ERR_UNSUPPORTED;
  const Range in[5] = {rng(x, size_t(T) * H * eb), rng(weight, size_t(V) * H * eb),
                       rng(target, size_t(T) * 8), rng(lse, size_t(T) * 4),
                       rng(grad_loss, reduction == FLCE_REDUCTION_NONE ? size_t(T) * 4 : 4)};
  const Range out[4] = {rng(grad_x, size_t(T) * H * eb), rng(grad_weight, size_t(V) * H * eb),
                        rng(workspace, need), rng(status, sizeof(int))};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 5; ++j)
      if (overlap(out[i], in[j])) return FLCE_ERR_ALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(out[i], out[j])) return FLCE_ERR_ALIAS;
  }

  flce::Device dev;
  int rc = check_device(&dev);
  if (rc != FLCE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  Carver c;
  c.base = static_cast<uint8_t*>(workspace);
  BwdWs w;
  carve_bwd(c, T, H, V, dtype, &w);
  const float scale = reduction == FLCE_REDUCTION_MEAN ? 1.0f / float(T) : 1.0f;
  const bool bf16 = dtype == FLCE_DTYPE_BF16;
  const auto DT = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const uint32_t bk = bf16 ? 64 : 32;  // elements per 128-byte swizzle row

  cudaError_t e = cudaSuccess;
  // Slab-invariant operand maps.
  CUtensorMap tx, tx_mn, txh, txl, txth, txtl;
  if (bf16) {
    if (!flce::make_tmap_2d(&tx, DT, x, H, T, H * 2, bk,
                            flce::core_a_box_rows(flce::role_core(dev.sms, FLCE_ROLE_DZ))) ||
        !flce::make_tmap_2d(&tx_mn, DT, x, H, T, H * 2, 64, 64))
      return FLCE_ERR_CUDA;
  } else {
    // B operands boxed for their role's core (128 rows per CTA on SM pairs, 256 on one SM)
    const uint32_t gbox = flce::core_b_box_rows(flce::tf32_core(dev.sms, FLCE_ROLE_GRADS));
    if (!flce::make_tmap_2d(&txh, DT, w.x_hi, H, T, H * 4, bk, kTileM) ||
        !flce::make_tmap_2d(&txl, DT, w.x_lo, H, T, H * 4, bk, kTileM) ||
        !flce::make_tmap_2d(&txth, DT, w.xt_hi, T, H, w.ldT * 4, bk, gbox) ||
        !flce::make_tmap_2d(&txtl, DT, w.xt_lo, T, H, w.ldT * 4, bk, gbox))
      return FLCE_ERR_CUDA;
    const float* xf = static_cast<const float*>(x);
    e = flce::launch_split_tf32(xf, T, H, H, w.x_hi, w.x_lo, false, s);
    if (e == cudaSuccess) e = flce::launch_split_tf32(xf, T, H, w.ldT, w.xt_hi, w.xt_lo, true, s);
    if (e != cudaSuccess) return FLCE_ERR_CUDA;
  }

  for (int64_t si = 0; si < w.n_slabs && e == cudaSuccess; ++si) {
    const int64_t slab0 = si * w.vc;
    const int64_t sw = (V - slab0) < w.vc ? (V - slab0) : w.vc;
    const int mode = w.n_slabs == 1 ? 0 : (si == 0 ? 1 : (si == w.n_slabs - 1 ? 3 : 2));

    flce::DzLaunch dz{};
    dz.target = target;
    dz.lse = lse;
    dz.row_scale = reduction == FLCE_REDUCTION_NONE ? grad_loss : nullptr;
    dz.dz = w.dz;
    dz.dz_lo = w.dz_lo;
    dz.dzt_hi = w.dzt_hi;
    dz.dzt_lo = w.dzt_lo;
    dz.ldz = int(w.vc);
    dz.ldt = int(w.ldT);
    dz.T = int(T);
    dz.H = int(H);
    dz.slab0 = int(slab0);
    dz.slab_w = int(sw);
    dz.status = status;
    dz.tile_counter = w.counter;
    dz.sms = dev.sms;
    dz.stream = s;

    flce::GradWLaunch gw{};
    gw.grad_w = grad_weight;
    gw.grad_loss = reduction == FLCE_REDUCTION_NONE ? nullptr : grad_loss;
    gw.scale = scale;
    gw.H = int(H);
    gw.T = int(T);
    gw.slab0 = int(slab0);
    gw.slab_w = int(sw);
    gw.status = status;
    gw.tile_counter = w.counter;
    gw.sms = dev.sms;
    gw.stream = s;

    flce::GradXLaunch gx{};
    gx.acc = bf16 ? w.acc : static_cast<float*>(grad_x);
    gx.grad_x = grad_x;
    gx.grad_loss = reduction == FLCE_REDUCTION_NONE ? nullptr : grad_loss;
    gx.scale = scale;
    gx.mode = mode;
    gx.T = int(T);
    gx.H = int(H);
    gx.K = int(sw);
    gx.status = status;
    gx.sms = dev.sms;
    gx.stream = s;

    if (bf16) {
      const uint8_t* wslab = static_cast<const uint8_t*>(weight) + size_t(slab0) * H * 2;
      CUtensorMap tws, tdz_mn, tdz_k, tw_mn;
      const uint32_t wbox = flce::core_b_box_rows(flce::role_core(dev.sms, FLCE_ROLE_DZ));
      const uint32_t dzbox = flce::core_a_box_rows(flce::role_core(dev.sms, FLCE_ROLE_GRADS));
      if (!flce::make_tmap_2d(&tws, DT, wslab, H, sw, H * 2, bk, wbox) ||
          !flce::make_tmap_2d(&tdz_mn, DT, w.dz, sw, T, w.vc * 2, 64, 64) ||
          !flce::make_tmap_2d(&tdz_k, DT, w.dz, sw, T, w.vc * 2, bk, dzbox) ||
          !flce::make_tmap_2d(&tw_mn, DT, wslab, H, sw, H * 2, 64, 64))
        return FLCE_ERR_CUDA;
      e = flce::timed_launch(1, s, [&] { return flce::launch_dz_bf16(tx, tws, dz); });
      if (e == cudaSuccess)
        e = flce::timed_launch(
            4, s, [&] { return flce::launch_grads_bf16(tdz_mn, tx_mn, tdz_k, tw_mn, gw, gx); });
    } else {
      // this slab's weight rows split into TF32 hi/lo, as rows [sw][H] and transposed [H][sw]
      const float* wslab = static_cast<const float*>(weight) + size_t(slab0) * H;
      e = flce::launch_split_tf32(wslab, sw, H, H, w.w_hi, w.w_lo, false, s);
      if (e == cudaSuccess)
        e = flce::launch_split_tf32(wslab, sw, H, w.ldVc, w.wt_hi, w.wt_lo, true, s);
      if (e != cudaSuccess) break;
      CUtensorMap twh, twl, tdzth, tdztl, tdzh, tdzl, twth, twtl;
      const uint32_t dbox = flce::core_b_box_rows(flce::tf32_core(dev.sms, FLCE_ROLE_DZ));
      const uint32_t gbox = flce::core_b_box_rows(flce::tf32_core(dev.sms, FLCE_ROLE_GRADS));
      if (!flce::make_tmap_2d(&twh, DT, w.w_hi, H, sw, H * 4, bk, dbox) ||
          !flce::make_tmap_2d(&twl, DT, w.w_lo, H, sw, H * 4, bk, dbox) ||
          !flce::make_tmap_2d(&tdzth, DT, w.dzt_hi, T, sw, w.ldT * 4, bk, kTileM) ||
          !flce::make_tmap_2d(&tdztl, DT, w.dzt_lo, T, sw, w.ldT * 4, bk, kTileM) ||
          !flce::make_tmap_2d(&tdzh, DT, w.dz, sw, T, w.vc * 4, bk, kTileM) ||
          !flce::make_tmap_2d(&tdzl, DT, w.dz_lo, sw, T, w.vc * 4, bk, kTileM) ||
          !flce::make_tmap_2d(&twth, DT, w.wt_hi, sw, H, w.ldVc * 4, bk, gbox) ||
          !flce::make_tmap_2d(&twtl, DT, w.wt_lo, sw, H, w.ldVc * 4, bk, gbox))
        return FLCE_ERR_CUDA;
      e = flce::timed_launch(1, s, [&] { return flce::launch_dz_tf32(txh, twh, txl, twl, dz); });
      if (e == cudaSuccess)
        e = flce::timed_launch(2, s, [&] { return flce::launch_gradw_tf32(tdzth, txth, tdztl, txtl, gw); });
      if (e == cudaSuccess)
        e = flce::timed_launch(3, s, [&] { return flce::launch_gradx_tf32(tdzh, twth, tdzl, twtl, gx); });
    }
  }
  return e == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}

int flce_forward_backward(const void* x, const void* weight, const int64_t* target, int64_t T,
                          int64_t H, int64_t V, int dtype, int reduction, const float* grad_loss,
                          float* loss, float* lse, void* grad_x, void* grad_weight,
                          void* workspace, size_t workspace_bytes, int* status, void* stream) {
  if (!x || !weight || !target || !grad_loss || !loss || !lse || !grad_x || !grad_weight ||
      !status)
    return FLCE_ERR_ARG;
  if (!dims_ok(T, H, V, dtype)) return FLCE_ERR_ARG;
  if (reduction != FLCE_REDUCTION_SUM && reduction != FLCE_REDUCTION_MEAN &&
      reduction != FLCE_REDUCTION_NONE)
    return FLCE_ERR_ARG;
  const int eb = elem_bytes(dtype);
  if ((H * eb) % 16 != 0 || !aligned16(x) || !aligned16(weight) || !aligned16(grad_x) ||
      !aligned16(grad_weight))
    return FLCE_ERR_UNSUPPORTED;
  const size_t need = flce_forward_backward_workspace_size(T, H, V, dtype);
  if (!workspace || workspace_bytes < need) return FLCE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return FLCE_ERR_UNSUPPORTED;
  const size_t per = reduction == FLCE_REDUCTION_NONE ? size_t(T) * 4 : 4;
  const Range in[4] = {rng(x, size_t(T) * H * eb), rng(weight, size_t(V) * H * eb),
                       rng(target, size_t(T) * 8), rng(grad_loss, per)};
  const Range out[6] = {rng(loss, per), rng(lse, size_t(T) * 4),
                        rng(grad_x, size_t(T) * H * eb), rng(grad_weight, size_t(V) * H * eb),
                        rng(workspace, need), rng(status, sizeof(int))};
  for (int i = 0; i < 6; ++i) {
    for (int j = 0; j < 4; ++j)
      if (overlap(out[i], in[j])) return FLCE_ERR_ALIAS;
    for (int j = i + 1; j < 6; ++j)
      if (overlap(out[i], out[j])) return FLCE_ERR_ALIAS;
  }
  if (!fused_schedule(T, dtype)) {
    int rc = flce_forward(x, weight, target, T, H, V, dtype, reduction, loss, lse, workspace,
                          workspace_bytes, status, stream);
    if (rc != FLCE_OK) return rc;
    return flce_backward(x, weight, target, lse, T, H, V, dtype, reduction, grad_loss, grad_x,
                         grad_weight, workspace, workspace_bytes, status, stream);
  }

  flce::Device dev;
  int rc = check_device(&dev);
  if (rc != FLCE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carver c;
  c.base = static_cast<uint8_t*>(workspace);
  FusedWs w;
  carve_fused(c, T, H, V, &w);
  const auto DT = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool none = reduction == FLCE_REDUCTION_NONE;
  CUtensorMap tw_k, tw_mn;
  const flce::Core fcore = flce::role_core(dev.sms, FLCE_ROLE_FORWARD);
  const flce::Core gcore = flce::role_core(dev.sms, FLCE_ROLE_GRADS);
  if (!flce::make_tmap_2d(&tw_k, DT, weight, H, V, H * 2, 64, flce::core_b_box_rows(fcore)) ||
      !flce::make_tmap_2d(&tw_mn, DT, weight, H, V, H * 2, 64, 64))
    return FLCE_ERR_CUDA;

  cudaError_t e = cudaSuccess;
  for (int64_t ci = 0; ci < w.n_chunks && e == cudaSuccess; ++ci) {
    const int64_t t0 = ci * w.rows;
    const int64_t rows = (T - t0) < w.rows ? (T - t0) : w.rows;
    const uint8_t* xc = static_cast<const uint8_t*>(x) + size_t(t0) * H * 2;
    CUtensorMap tx_k, tx_mn, tz_k, tz_mn;
    if (!flce::make_tmap_2d(&tx_k, DT, xc, H, rows, H * 2, 64, flce::core_a_box_rows(fcore)) ||
        !flce::make_tmap_2d(&tx_mn, DT, xc, H, rows, H * 2, 64, 64) ||
        !flce::make_tmap_2d(&tz_k, DT, w.zbuf, V, rows, w.ldz * 2, 64,
                            flce::core_a_box_rows(gcore)) ||
        !flce::make_tmap_2d(&tz_mn, DT, w.zbuf, V, rows, w.ldz * 2, 64, 64))
      return FLCE_ERR_CUDA;
    flce::ChunkLaunch cl{};
    cl.target = target + t0;
    cl.lse = lse + t0;
    cl.row_scale = none ? grad_loss + t0 : nullptr;
    cl.grad_loss = none ? nullptr : grad_loss;
    cl.scale = reduction == FLCE_REDUCTION_MEAN ? 1.0f / float(T) : 1.0f;
    cl.zbuf = w.zbuf;
    cl.ldz = int(w.ldz);
    cl.part_m = w.part_m;
    cl.part_s = w.part_s;
    cl.zy = w.zy;
    cl.sx = w.sx;
    cl.grad_x_rows = static_cast<uint8_t*>(grad_x) + size_t(t0) * H * 2;
    cl.grad_w = grad_weight;
    cl.gw_mode = ci == 0 ? 0 : 4;  // written by the first chunk, summed in place after it
    cl.tile_counter = w.counter;
    cl.rows = int(rows);
    cl.H = int(H);
    cl.V = int(V);
    cl.status = status;
    cl.sms = dev.sms;
    cl.stream = s;
    e = flce::timed_launch(0, s, [&] { return flce::launch_chunk_logits(tx_k, tw_k, cl); });
    if (e == cudaSuccess)
      e = flce::launch_combine_rows(w.part_m, w.part_s, w.zy, w.sx, target + t0, int(rows),
                                    int(V), int(w.ldz / (kTileN / 2)), kTileN / 2, lse + t0,
                                    w.block_sums + t0 / flce::kLossBlockTokens,
                                    none ? loss + t0 : nullptr, status,
                                    s);
    if (e == cudaSuccess) e = flce::launch_form_dz(cl);
    if (e == cudaSuccess)
      e = flce::timed_launch(4, s,
                             [&] { return flce::launch_chunk_grads(tz_k, tw_mn, tz_mn, tx_mn, cl); });
  }
  if (e == cudaSuccess && !none)
    e = flce::launch_finalize(w.block_sums, int(cdiv(T, flce::kLossBlockTokens)), int(T),
                              reduction, loss, s);
  return e == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}

}  // extern "C"
