// flce_fused.cu - forward and backward in one call, over chunks of tokens, without recomputing
// the logits. The Liger schedule discussed in "[example] fused_linear_cross_entropy kernel"
// (Helion PR #1268) produces the gradients while the forward runs, and "feat(FLCE): add helion
// version of fused linear cross entropy" (Liger-Kernel PR #928) describes its chunked backward,
// which computes each chunk's logits again before accumulating both gradients; here a chunk's
// logits are computed once and kept for its backward.
//
// Per chunk of Tc tokens (never all T: the chunk buffer holds at most half the tokens' logits):
//   1. logits  : z = x_c . W^T (tcgen05), kept as bf16 z - m (m: the maximum of each 128-column
//                half-tile) plus lse partials per half-tile (LogitsEpi)
//   2. combine : lse, per-token loss / loss block sums of the chunk rows (k_fwd_combine)
//   3. form dz : dz = (exp(z - lse) - onehot) * row scale, in place, bf16 (k_form_dz)
//   4. grads   : grad_x[chunk] = dz . W (complete, K = V) and grad_W (+)= dz^T . x_c (K = Tc),
//                one launch, dynamic tiles; grad_W is written by the first chunk and summed in
//                place, in its bf16 output, by the later ones (in chunk order)
// FLOPs: 6 T H V (forward + two gradient contractions) instead of 8 T H V with recompute.
#include <algorithm>

#include "epilogues.cuh"
#include "flce_internal.h"
#include "gemm_pair.cuh"

namespace flce {

// dz[t][v] = (exp(zbuf[t][v] + m[v / 128][t] - lse[t]) - [v == target[t]]) * row_scale[t] for
// v < V, 0 for V <= v < ldz; 8 consecutive columns (16 bytes) per thread, in place. (m holds
// one shift per 128-column half-tile, as LogitsEpi stored the logits.)
__global__ void __launch_bounds__(256)
    k_form_dz(__nv_bfloat16* __restrict__ zbuf, int ldz, int rows, int V,
              const float* __restrict__ part_m, const float* __restrict__ lse,
              const int64_t* __restrict__ target, const float* __restrict__ row_scale) {
  const int vecs = ldz / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(rows) * vecs) return;
  const int t = static_cast<int>(idx / vecs);
  const int v0 = static_cast<int>(idx - static_cast<int64_t>(t) * vecs) * 8;
  uint4* p = reinterpret_cast<uint4*>(zbuf + static_cast<size_t>(t) * ldz + v0);
  const float off = (part_m[static_cast<size_t>(v0 / 128) * rows + t] - lse[t]) * kLog2e;
  const long long y = static_cast<long long>(target[t]);
  const float rs = row_scale ? row_scale[t] : 1.0f;
  uint4 w = *p;
  uint32_t* u = reinterpret_cast<uint32_t*>(&w);
  float d[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = __uint_as_float(u[j] << 16);
    const float hi = __uint_as_float(u[j] & 0xffff0000u);
    d[2 * j] = lo;
    d[2 * j + 1] = hi;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int v = v0 + j;
    float e = ex2(fmaf(d[j], kLog2e, off));
    if (v == y) e -= 1.0f;
    d[j] = v < V ? e * rs : 0.0f;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) u[j] = pack_bf16x2(d[2 * j], d[2 * j + 1]);
  *p = w;
}

cudaError_t launch_chunk_logits(const CUtensorMap& tx_c, const CUtensorMap& tw,
                                const ChunkLaunch& c) {
  LogitsEpi::Args ea{c.target, c.part_m, c.part_s, c.zy, c.sx, c.zbuf, c.ldz, c.rows, c.V};
  const Core core = role_core(c.sms, FLCE_ROLE_FORWARD);  // maps boxed for this core
  GemmGrid g{};
  // token-row raster: the chunk's x rows stay in L2 while W streams past, in one group when
  // they fit in kChunkRowsL2Bytes (then each W tile is read from DRAM once per chunk, by the
  // tiles of all the chunk's rows in the same wave), else in groups of that size
  const int tile_rows = core_tile_rows(core);
  g.p[0] = make_problem(c.rows, c.V, c.H, 64, false, false, tile_rows, 0, false);
  const int64_t tile_x_bytes = static_cast<int64_t>(tile_rows) * c.H * 2;
  const int fit = static_cast<int>(std::max<int64_t>(1, kChunkRowsL2Bytes / tile_x_bytes));
  g.p[0].group_m = std::max(g.p[0].group_m, std::min(g.p[0].m_tiles, fit));
  g.num_problems = 1;
  g.status = c.status;
  g.tile_counter = c.tile_counter;  // tiles in list order: the pairs sharing a W tile stay in step
  if (core != kCoreSingle)
    return launch_pair_core<LogitsEpi, NoEpi, 2>(core, tx_c, tw, tx_c, tw, g, ea, NoEpi::Args{},
                                                 c.sms, c.stream, FLCE_ROLE_FORWARD);
  return launch_gemm<false, LogitsEpi, NoEpi>(tx_c, tw, tx_c, tw, g, ea, NoEpi::Args{}, c.sms,
                                              c.stream);
}

cudaError_t launch_form_dz(const ChunkLaunch& c) {
  const int64_t n = static_cast<int64_t>(c.rows) * (c.ldz / 8);
  const int64_t blocks = (n + 255) / 256;
  k_form_dz<<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(
      c.zbuf, c.ldz, c.rows, c.V, c.part_m, c.lse, c.target, c.row_scale);
  return cudaGetLastError();
}

// grad_x rows of the chunk (A = dz K-major, B = W MN-major, K = V: few long tiles, listed
// first) and grad_W (A = dz MN-major, B = x_c MN-major, K = Tc: many short tiles) in one launch
// whose CTAs (or CTA pairs) take tiles from a shared counter, longest first, so the long tiles
// spread evenly.
cudaError_t launch_chunk_grads(const CUtensorMap& tz_k, const CUtensorMap& tw_mn,
                               const CUtensorMap& tz_mn, const CUtensorMap& tx_mn,
                               const ChunkLaunch& c) {
  typename GradXEpi<false>::Args ex{nullptr, c.grad_x_rows, c.grad_loss, c.scale,
                                    c.rows,  c.H,           0};
  typename GradXEpi<false>::Args ew{nullptr, c.grad_w, c.grad_loss, c.scale,
                                    c.V,     c.H,      c.gw_mode};
  const Core core = role_core(c.sms, FLCE_ROLE_GRADS);  // zbuf K-major map boxed to match
  const int tile_rows = core_tile_rows(core);
  GemmGrid g{};
  g.p[0] = make_problem(c.rows, c.H, c.V, 64, false, true, tile_rows, 0);
  g.p[1] = make_problem(c.V, c.H, c.rows, 64, true, true, tile_rows,
                        g.p[0].m_tiles * g.p[0].n_tiles);
  g.num_problems = 2;
  g.status = c.status;
  g.tile_counter = c.tile_counter;
  if (core != kCoreSingle)
    return launch_pair_core<GradXEpi<false>, GradXEpi<false>>(core, tz_k, tw_mn, tz_mn, tx_mn, g, ex,
                                                              ew, c.sms, c.stream,
                                                              FLCE_ROLE_GRADS);
  return launch_gemm<false, GradXEpi<false>, GradXEpi<false>>(tz_k, tw_mn, tz_mn, tx_mn, g, ex, ew,
                                                              c.sms, c.stream);
}

}  // namespace flce
