// flce_fwd.cu - forward kernels: the fused projection + online log-sum-exp contraction, the
// fixed-order merge of its per-vocab-tile partials into lse[T], and the deterministic loss
// reduction.
#include "epilogues.cuh"
#include "flce_internal.h"
#include "gemm_pair.cuh"

namespace flce {

// The combine kernel: a block of 8 warps per 32 tokens; warp w merges the partials of the
// w-th eighth of the vocab tiles for those tokens (lane = token, so every load of a tile's
// partials is 32 consecutive tokens), then warp 0 merges the eight results in warp order.
constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = 32 * kCombineWarps;
constexpr int kCombineTokens = kLossBlockTokens;  // tokens per block and per loss block sum

// One partial into the running (M, S, SX): S sums exp(z - M) over every column seen, SX over
// every column but the target.
__device__ __forceinline__ void lse_merge(float& M, float& S, float& SX, float m, float s,
                                          float s_x) {
  const float mn = fmaxf(M, m);
  const float f0 = ex2((M - mn) * kLog2e), f1 = ex2((m - mn) * kLog2e);
  S = S * f0 + s * f1;
  SX = SX * f0 + s_x * f1;
  M = mn;
}

// Merge the per-(vocab tile) partials of each token in a fixed order (eighths of the tile
// range, each in increasing tile order, then the eighths in order):
//   M = max_i m_i,  S = sum_i s_i exp(m_i - M),  lse = M + ln S,
// and, with the target tile's sum taken without the target column (sx), the same merge SX of
// the terms of every column but the target. The per-token loss l = lse - z[t, target[t]] is
// formed as ln(1 + SX) when the target logit is the row maximum (then lse and z[t, target[t]]
// nearly cancel and l is close to 0), else as (M - z[t, target[t]]) + ln S.
// Writes lse[t] and one partial loss sum per 32 tokens (fixed-order shuffle tree); with
// per_token non-null (the 'none' reduction) it also writes l[t] there. tile_cols: vocab columns
// per partial.
__global__ void __launch_bounds__(kCombineThreads)
    k_fwd_combine(const float* __restrict__ part_m, const float* __restrict__ part_s,
                  const float* __restrict__ zy, const float* __restrict__ sx,
                  const int64_t* __restrict__ target, int T, int V, int n_tiles, int tile_cols,
                  float* __restrict__ lse, float* __restrict__ block_sums,
                  float* __restrict__ per_token, int* status) {
  __shared__ float3 partial[kCombineWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kCombineTokens + lane;
  const bool valid = t < T;
  const int64_t y = valid ? target[t] : -1;
  const bool in_range = y >= 0 && y < V;
  const int ty = in_range ? static_cast<int>(y / tile_cols) : -1;
  const int per_warp = (n_tiles + kCombineWarps - 1) / kCombineWarps;
  const int i0 = warp * per_warp;
  const int i1 = min(n_tiles, i0 + per_warp);
  float M = -INFINITY, S = 0.f, SX = 0.f;
  if (valid) {
    const float sxt = (ty >= i0 && ty < i1) ? sx[t] : 0.f;
    for (int i = i0; i < i1; ++i) {
      const float m = part_m[static_cast<size_t>(i) * T + t];
      const float s = part_s[static_cast<size_t>(i) * T + t];
      if (m == -INFINITY) continue;  // an empty partial (a half-tile wholly beyond V)
      lse_merge(M, S, SX, m, s, i == ty ? sxt : s);
    }
  }
  partial[warp][lane] = make_float3(M, S, SX);
  __syncthreads();
  if (warp != 0) return;
  M = -INFINITY;
  S = 0.f;
  SX = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    const float3 p = partial[w][lane];
    if (p.x != -INFINITY) lse_merge(M, S, SX, p.x, p.y, p.z);
  }
  float l = 0.f;
  if (valid) {
    const float lnS = logf(S);
    lse[t] = M + lnS;
    if (!in_range) {
      atomicOr(status, FLCE_STATUS_TARGET_RANGE);
      l = __int_as_float(0x7fc00000);  // NaN
    } else {
      const float z_y = zy[t];
      l = z_y == M ? log1pf(SX) : (M - z_y) + lnS;
    }
    if (per_token) per_token[t] = l;
  }
  // Fixed-order reduction of the block's 32 per-token losses.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_down_sync(0xffffffffu, l, o);
  if (lane == 0) block_sums[blockIdx.x] = l;
}

// loss = sum of the block sums (fp64, fixed order), divided by T for the mean reduction.
__global__ void __launch_bounds__(256)
    k_fwd_finalize(const float* __restrict__ block_sums, int n, int T, int reduction,
                   float* __restrict__ loss) {
  __shared__ double part[256];
  double acc = 0.0;
  for (int i = threadIdx.x; i < n; i += 256) acc += static_cast<double>(block_sums[i]);
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double total = part[0];
    if (reduction == FLCE_REDUCTION_MEAN) total /= static_cast<double>(T);
    loss[0] = static_cast<float>(total);
  }
}

// Projection + online log-sum-exp over the (token tile, vocab tile) pairs of vocab columns
// [col0, col0 + cols) (W maps cover those rows only).
template <bool kTF32>
static cudaError_t launch_projection(const CUtensorMap& tx, const CUtensorMap& tw,
                                     const CUtensorMap& tx_lo, const CUtensorMap& tw_lo,
                                     const FwdLaunch& p, int col0, int cols) {
  // bf16: single-SM tiles here (the pair cores launch from launch_forward_bf16); fp32: the
  // core tf32_core picks, for which the W maps are boxed
  const Core core = kTF32 ? tf32_core(p.sms, FLCE_ROLE_FORWARD) : kCoreSingle;
  GemmGrid g{};
  g.p[0] = make_problem(p.T, cols, p.H, StageGeom<kTF32>::kBK, false, false, core_tile_rows(core),
                        0, true);
  g.num_problems = 1;
  g.status = p.status;
  g.tile_counter = p.tile_counter;
  FwdEpi::Args ea{p.target, p.part_m, p.part_s, p.zy, p.sx, p.T, cols, col0};
  if constexpr (kTF32) {
    if (core == kCorePair)
      return launch_pair_tf32<FwdEpi>(tx, tw, tx_lo, tw_lo, g, ea, p.sms, p.stream);
  }
  return launch_gemm<kTF32, FwdEpi, NoEpi>(tx, tw, tx_lo, tw_lo, g, ea, NoEpi::Args{}, p.sms,
                                           p.stream);
}

// The combine (lse, per-token loss, block sums) and finalize kernels after the projection.
cudaError_t launch_forward_combine(const FwdLaunch& p) {
  const int n_tiles = (p.V + kBN - 1) / kBN;
  const bool none = p.reduction == FLCE_REDUCTION_NONE;
  cudaError_t e = launch_combine_rows(p.part_m, p.part_s, p.zy, p.sx, p.target, p.T, p.V,
                                      n_tiles, kBN, p.lse, p.block_sums, none ? p.loss : nullptr,
                                      p.status, p.stream);
  if (e != cudaSuccess || none) return e;
  return launch_finalize(p.block_sums, (p.T + kCombineTokens - 1) / kCombineTokens, p.T,
                         p.reduction, p.loss, p.stream);
}

cudaError_t launch_combine_rows(const float* part_m, const float* part_s, const float* zy,
                                const float* sx, const int64_t* target, int rows, int V,
                                int n_tiles, int tile_cols, float* lse, float* block_sums,
                                float* per_token, int* status, cudaStream_t stream) {
  const int nblk = (rows + kCombineTokens - 1) / kCombineTokens;
  k_fwd_combine<<<nblk, kCombineThreads, 0, stream>>>(part_m, part_s, zy, sx, target, rows, V,
                                                      n_tiles, tile_cols, lse, block_sums,
                                                      per_token, status);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* block_sums, int n_blocks, int T, int reduction,
                            float* loss, cudaStream_t stream) {
  k_fwd_finalize<<<1, 256, 0, stream>>>(block_sums, n_blocks, T, reduction, loss);
  return cudaGetLastError();
}

cudaError_t launch_forward_bf16(const CUtensorMap& tx, const CUtensorMap& tw, const FwdLaunch& p) {
  const Core core = role_core(p.sms, FLCE_ROLE_FORWARD);
  if (core != kCoreSingle) {  // x boxed {64 x core_a_box_rows}, W {64 x 128} for this path
    GemmGrid g{};
    g.p[0] = make_problem(p.T, p.V, p.H, 64, false, false, core_tile_rows(core), 0, true);
    g.num_problems = 1;
    g.status = p.status;
    g.tile_counter = p.tile_counter;
    FwdEpi::Args ea{p.target, p.part_m, p.part_s, p.zy, p.sx, p.T, p.V, 0};
    cudaError_t e = launch_pair_core<FwdEpi, NoEpi, 2>(core, tx, tw, tx, tw, g, ea, NoEpi::Args{},
                                                       p.sms, p.stream, FLCE_ROLE_FORWARD);
    if (e != cudaSuccess) return e;
    return launch_forward_combine(p);
  }
  cudaError_t e = launch_projection<false>(tx, tw, tx, tw, p, 0, p.V);
  if (e != cudaSuccess) return e;
  return launch_forward_combine(p);
}

cudaError_t launch_forward_tf32(const CUtensorMap& tx_hi, const CUtensorMap& tw_hi,
                                const CUtensorMap& tx_lo, const CUtensorMap& tw_lo,
                                const FwdLaunch& p, int col0, int cols) {
  return launch_projection<true>(tx_hi, tw_hi, tx_lo, tw_lo, p, col0, cols);
}

}  // namespace flce
