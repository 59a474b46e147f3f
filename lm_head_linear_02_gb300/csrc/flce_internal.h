// flce_internal.h - host-side declarations shared by the libflce translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/flce.h"

namespace flce {

// Tile sizes of the contraction core (see gemm.cuh).
constexpr int kTileM = 128;
constexpr int kTileN = 256;

// Process-wide tuning values (set through flce_set_tuning; read at each launch).
//   tune_raster_rows(): rows of the M dimension per raster group (tiles walk N inside a group,
//                       so the group's A rows stay in L2 while B streams); default 2048.
//   tune_sm_pairs():    bit mask of the bf16 roles (FLCE_ROLE_*) that run on CTA pairs, or -1
//                       (the default) to decide per device.
//   tune_wide_tiles(): bit mask of the roles whose CTA pairs use 256-row CTA tiles, or -1 (the
//                      default: kDefaultWideRoles).
//   tune_raster_vocab(): vocabulary rows per raster group of the forward projection and the
//                       backward's dz launches (whose N dimension is the vocabulary): tiles walk
//                       the token rows inside a group, so the group's weight rows stay in L2
//                       while x streams; 0 rasters those over token rows too.
//   tune_split_epilogue(): bit mask of the roles (FLCE_ROLE_FORWARD: the forward projection and
//                       the chunk logits; FLCE_ROLE_DZ) whose wide pair tiles drain each row
//                       block with two epilogue warps (16 per CTA) instead of one.
int tune_raster_rows();
int tune_raster_vocab();
int tune_split_epilogue();
//   tune_ordered_drain(): bit mask of the roles whose wide pair tiles (one epilogue warp per row
//                       block) drain their two 128-row halves one after the other, so that the
//                       next tile's MMAs on the first half overlap the drain of the second.
int tune_ordered_drain();
int tune_sm_pairs();
int tune_wide_tiles();

// Consumes a pending flce_test_withhold_signal() request (true at most once per request).
bool take_withhold_request();

// Roles measured faster on CTA pairs, used by the automatic choice when every SM of the device
// can be paired: all three (with the wide CTA tiles below; on 128-row CTA tiles dz alone was
// faster on single SMs).
constexpr int kAutoPairRoles = FLCE_ROLE_FORWARD | FLCE_ROLE_DZ | FLCE_ROLE_GRADS;

// Default of tune_raster_vocab(): groups of 4096 weight rows (32 MB at H = 4096). Measured on
// GB300 at T = 16384, V = 128256: the forward read 5.7 instead of 8.6 GB of DRAM per launch and
// dz 1.9 instead of 2.3 GB per slab, and the step ran 0.7-0.8% faster than with the 2048-row
// token raster; groups of 6144 and 8192 rows re-read more (L2 no longer holds the group while x
// streams past) and ran no faster.
constexpr int kDefaultRasterVocab = 4096;

// Token rows of a single-call chunk kept in L2 as one raster group of its logits launch
// (46 MB for 5632 rows at H = 4096).
constexpr int64_t kChunkRowsL2Bytes = int64_t(48) << 20;

// Default bf16 chunk-logits budget of the single call (FLCE_TUNE_CHUNK_BYTES): 1.5 GiB.
constexpr int64_t kDefaultChunkBytes = int64_t(3) << 29;

// Default of tune_split_epilogue(): none. Measured on GB300 at the headline size and on the
// Llama-2 head: two epilogue warps per row block left the tensor pipe's active cycles where
// they were (dz 85.8% -> 85.2%, forward 89.3% -> 89.4%) and the launches 0.3% slower.
constexpr int kDefaultSplitEpilogue = 0;

// Default of tune_ordered_drain(): the forward projection (and the single call's chunk logits)
// and dz, whose K = H main loops are short enough for the drain to matter. Measured on GB300
// at T = 16384, H = 4096, V = 128256 against draining both halves together: a tile's period
// (SM clock stamps per tile) 1.4% shorter for the forward and 2.3% for dz; in the power-capped
// step the forward launch 0.6% and dz 1.4% faster, the step 0.3-0.5%; the single call's chunk
// logits (forward role) 1.4% faster (three interleaved runs each). The gradient launch
// (K = 16384 or 32256) loses: its epilogue's accumulator traffic during the next tile's main
// loop made its tiles 3% longer.
constexpr int kDefaultOrderedDrain = FLCE_ROLE_FORWARD | FLCE_ROLE_DZ;

// Roles measured faster on 256-row CTA tiles when they run on CTA pairs.
constexpr int kDefaultWideRoles = FLCE_ROLE_FORWARD | FLCE_ROLE_DZ | FLCE_ROLE_GRADS;

// Effective FLCE_ROLE_* mask of bf16 roles that run on CTA pairs on the current device.
int pair_roles(int sms);

// The contraction core a bf16 role launches on: single-SM 128 x 256 tiles, CTA pairs with
// 128-row CTA tiles (256 x 256 pair tiles) or CTA pairs with 256-row CTA tiles (512 x 256).
enum Core { kCoreSingle = 0, kCorePair = 1, kCoreWide = 2 };
inline Core role_core(int sms, int role) {
  if ((pair_roles(sms) & role) == 0) return kCoreSingle;
  const int w = tune_wide_tiles();
  return ((w >= 0 ? w : kDefaultWideRoles) & role) ? kCoreWide : kCorePair;
}
// The contraction core an fp32 (3xTF32) role launches on: CTA pairs with 128-row CTA tiles
// (256 x 256 pair tiles) when the role runs on SM pairs, else single-SM 128 x 256 tiles.
inline Core tf32_core(int sms, int role) {
  return (pair_roles(sms) & role) != 0 ? kCorePair : kCoreSingle;
}
// M rows of one tile (GemmProblem tile_rows) on a core.
inline int core_tile_rows(Core c) { return c == kCoreWide ? 512 : c == kCorePair ? 256 : 128; }
// Rows of the box of a K-major A operand map ({64 x rows}) on a core.
inline uint32_t core_a_box_rows(Core c) { return c == kCoreWide ? 256u : 128u; }
// Rows of the box of a K-major B operand map ({64 x rows}): one CTA's N half on pairs.
inline uint32_t core_b_box_rows(Core c) { return c == kCoreSingle ? 256u : 128u; }

struct Device {
  int id = -1;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
};

// Device properties of the current device (cached per device id). Returns false on CUDA error.
bool current_device(Device* d);

// 2-D tensor map with 128-byte swizzle, zero fill outside [0,inner) x [0,outer).
//   base: global address (16-byte aligned), inner/outer: extents in elements / rows,
//   row_bytes: stride between rows (multiple of 16), box_inner x box_outer: box in elements.
bool make_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t inner,
                  uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// ---------------------------------------------------------------- forward launchers (flce_fwd.cu)
struct FwdLaunch {
  const int64_t* target;
  float* part_m;      // [n_tiles][T]
  float* part_s;      // [n_tiles][T]
  float* zy;          // [T]
  float* sx;          // [T]: the target tile's exp-sum without the target column
  float* block_sums;  // [ceil(T / kLossBlockTokens)]
  float* lse;         // [T]
  float* loss;        // [1], or [T] for the 'none' reduction
  int* tile_counter;  // zeroed before the projection launch: tiles handed out in list order
  int* status;
  int T, H, V, reduction;
  int sms;
  cudaStream_t stream;
};
// bf16: projection over all V columns, then the combine. x/W maps: K-major boxes sized for the
// forward role's core.
cudaError_t launch_forward_bf16(const CUtensorMap& tx, const CUtensorMap& tw, const FwdLaunch& p);
// tf32: the projection over vocab columns [col0, col0 + cols) only (col0 a multiple of 256);
// the W maps (hi/lo, K-major {32 x 256}) cover those rows. launch_forward_combine follows the
// last one.
cudaError_t launch_forward_tf32(const CUtensorMap& tx_hi, const CUtensorMap& tw_hi,
                                const CUtensorMap& tx_lo, const CUtensorMap& tw_lo,
                                const FwdLaunch& p, int col0, int cols);
cudaError_t launch_forward_combine(const FwdLaunch& p);

// Tokens per loss block sum written by the combine kernel (chunks of the single call start at
// multiples of 256 tokens, so at multiples of this).
constexpr int kLossBlockTokens = 32;
// Merge the per-vocab-tile partials of `rows` tokens (all pointers already offset to those rows;
// tile_cols vocab columns per partial) into lse, one loss sum per kLossBlockTokens rows
// (block_sums) and, if per_token is non-null, l[t].
cudaError_t launch_combine_rows(const float* part_m, const float* part_s, const float* zy,
                                const float* sx, const int64_t* target, int rows, int V,
                                int n_tiles, int tile_cols, float* lse, float* block_sums,
                                float* per_token, int* status, cudaStream_t stream);
// loss[0] = sum of n_blocks block sums (fp64, fixed order), / T for the mean reduction.
cudaError_t launch_finalize(const float* block_sums, int n_blocks, int T, int reduction,
                            float* loss, cudaStream_t stream);

// ---------------------------------------------------------------- backward launchers (flce_bwd.cu)
struct DzLaunch {
  const int64_t* target;
  const float* lse;
  const float* row_scale;  // per-token upstream gradient ('none' reduction) or null
  void* dz;           // (softmax - onehot): bf16 [T][ldz] or fp32 hi [T][ldz]
  void* dz_lo;        // fp32 lo [T][ldz] (tf32 path)
  void* dzt_hi;       // fp32 [Vc][ldt] transposed hi (tf32 path)
  void* dzt_lo;       // fp32 [Vc][ldt] transposed lo (tf32 path)
  int ldz, ldt;
  int T, H, slab0, slab_w;
  int* tile_counter;  // or null (static schedule)
  int* status;
  int sms;
  cudaStream_t stream;
};
cudaError_t launch_dz_bf16(const CUtensorMap& tx, const CUtensorMap& tw_slab, const DzLaunch& p);
cudaError_t launch_dz_tf32(const CUtensorMap& tx_hi, const CUtensorMap& tw_hi,
                           const CUtensorMap& tx_lo, const CUtensorMap& tw_lo, const DzLaunch& p);

struct GradWLaunch {
  void* grad_w;  // [V][H] (dtype); rows slab0 .. slab0 + slab_w are written
  const float* grad_loss;  // null for the 'none' reduction (g = scale = 1)
  float scale;   // 1 (sum, none) or 1/T (mean); g = grad_loss[0] * scale
  int H, T, slab0, slab_w;
  int* tile_counter;  // or null (static schedule); the bf16 launch of both gradients uses it
  int* status;
  int sms;
  cudaStream_t stream;
};
// tf32: A = dz^T slab (K-major, hi/lo), B = x^T (K-major, hi/lo).
cudaError_t launch_gradw_tf32(const CUtensorMap& tdzt_hi, const CUtensorMap& txt_hi,
                              const CUtensorMap& tdzt_lo, const CUtensorMap& txt_lo,
                              const GradWLaunch& p);

struct GradXLaunch {
  float* acc;    // fp32 [T][H] accumulator (bf16 path) or the fp32 output itself
  void* grad_x;  // [T][H] (dtype)
  const float* grad_loss;
  float scale;
  int mode;      // 0 only slab, 1 first, 2 middle, 3 last
  int T, H, K;
  int* status;
  int sms;
  cudaStream_t stream;
};
// bf16, one launch (on the role's core) for both gradients of a slab, longer-K problem first:
//   grad_W: A = dz slab (MN-major boxes {64 x 64}), B = x (MN-major boxes {64 x 64});
//   grad_x: A = dz slab (K-major {64 x core_a_box_rows}), B = W slab (MN-major {64 x 64}).
cudaError_t launch_grads_bf16(const CUtensorMap& tdz_mn, const CUtensorMap& tx_mn,
                              const CUtensorMap& tdz_k, const CUtensorMap& tw_mn,
                              const GradWLaunch& pw, const GradXLaunch& px);
// tf32: A = dz slab (K-major hi/lo), B = W^T slab (K-major hi/lo).
cudaError_t launch_gradx_tf32(const CUtensorMap& tdz_hi, const CUtensorMap& twt_hi,
                              const CUtensorMap& tdz_lo, const CUtensorMap& twt_lo,
                              const GradXLaunch& p);

// ---------------------------------------------------------------- single-call fwd+bwd (flce_fused.cu)
struct ChunkLaunch {
  const int64_t* target;   // chunk rows
  float* lse;              // chunk rows
  const float* row_scale;  // per-token upstream gradient of the chunk rows ('none') or null
  const float* grad_loss;  // global upstream gradient (sum/mean) or null ('none')
  float scale;             // 1 or 1/T
  __nv_bfloat16* zbuf;     // [rows][ldz] chunk logits (shifted) / dz
  int ldz;
  float *part_m, *part_s, *zy, *sx;  // [ldz / 128][rows] (one per half-tile) x 2, [rows] x 2
  void* grad_x_rows;       // grad_x + t0 * H
  void* grad_w;
  int gw_mode;             // 0: the first chunk writes grad_w, 4: later chunks add to it
  int* tile_counter;
  int rows, H, V;
  int* status;
  int sms;
  cudaStream_t stream;
};
// logits of the chunk: x_c K-major {64 x 128}, W K-major {64 x 256} ({64 x 128} when the forward
// role runs on SM pairs)
cudaError_t launch_chunk_logits(const CUtensorMap& tx_c, const CUtensorMap& tw,
                                const ChunkLaunch& c);
cudaError_t launch_form_dz(const ChunkLaunch& c);
// grads: dz K-major {64 x 128} and W MN-major {64 x 64}; dz MN-major and x_c MN-major {64 x 64}
cudaError_t launch_chunk_grads(const CUtensorMap& tz_k, const CUtensorMap& tw_mn,
                               const CUtensorMap& tz_mn, const CUtensorMap& tx_mn,
                               const ChunkLaunch& c);

// fp32 -> (hi, lo) TF32 split, optionally transposed: src [rows][cols] -> hi/lo [rows][ld_out]
// or, with transpose, hi/lo [cols][ld_out] (ld_out >= rows).
cudaError_t launch_split_tf32(const float* src, int64_t rows, int64_t cols, int64_t ld_out,
                              float* hi, float* lo, bool transpose, cudaStream_t stream);

}  // namespace flce
