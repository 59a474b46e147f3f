// flce_bwd.cu - backward kernels, one vocab slab [slab0, slab0 + slab_w) at a time:
//   dz     : recompute z = x . W_slab^T and form dz = (softmax - onehot) * g  (slab buffer)
//   grad_W : grad_W[slab] = dz_slab^T . x                                     (K = T, complete)
//   grad_x : grad_x (+)= dz_slab . W_slab                                     (split-K over slabs)
// plus the TF32 hi/lo operand split used by the fp32 path.
#include <atomic>

#include "epilogues.cuh"
#include "flce_internal.h"
#include "gemm_pair.cuh"

namespace flce {

// One problem M x N x K with K-major operands: bf16 on the single-CTA core; fp32 (3xTF32, hi
// and lo maps) on the core tf32_core(sms, role) picks, whose B maps are boxed for it.
template <bool kTF32, class Epi>
static cudaError_t run_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ta_lo,
                            const CUtensorMap& tb_lo, int M, int N, int K, int* status, int sms,
                            cudaStream_t stream, const typename Epi::Args& ea,
                            bool vocab_n = false, int role = 0) {
  const Core core = kTF32 ? tf32_core(sms, role) : kCoreSingle;
  GemmGrid g{};
  g.p[0] = make_problem(M, N, K, StageGeom<kTF32>::kBK, false, false, core_tile_rows(core), 0,
                        vocab_n);
  g.num_problems = 1;
  g.status = status;
  if constexpr (kTF32) {
    if (core == kCorePair) return launch_pair_tf32<Epi>(ta, tb, ta_lo, tb_lo, g, ea, sms, stream);
  }
  return launch_gemm<kTF32, Epi, NoEpi>(ta, tb, ta_lo, tb_lo, g, ea, NoEpi::Args{}, sms, stream);
}

cudaError_t launch_dz_bf16(const CUtensorMap& tx, const CUtensorMap& tw_slab, const DzLaunch& p) {
  typename DzEpi<false>::Args ea{p.target, p.lse, p.row_scale, p.dz, nullptr, nullptr, nullptr,
                                 p.ldz,    p.ldt, p.T,         p.slab0, p.slab_w};
  const Core core = role_core(p.sms, FLCE_ROLE_DZ);
  if (core != kCoreSingle) {  // x boxed {64 x core_a_box_rows}, W slab {64 x 128} for this path
    GemmGrid g{};
    g.p[0] = make_problem(p.T, p.slab_w, p.H, 64, false, false, core_tile_rows(core), 0, true);
    g.num_problems = 1;
    g.status = p.status;
    g.tile_counter = p.tile_counter;
    return launch_pair_core<DzEpi<false>, NoEpi, 2>(core, tx, tw_slab, tx, tw_slab, g, ea,
                                                    NoEpi::Args{}, p.sms, p.stream, FLCE_ROLE_DZ);
  }
  return run_gemm<false, DzEpi<false>>(tx, tw_slab, tx, tw_slab, p.T, p.slab_w, p.H, p.status,
                                       p.sms, p.stream, ea, true);
}

cudaError_t launch_dz_tf32(const CUtensorMap& tx_hi, const CUtensorMap& tw_hi,
                           const CUtensorMap& tx_lo, const CUtensorMap& tw_lo, const DzLaunch& p) {
  typename DzEpi<true>::Args ea{p.target,
                                p.lse,
                                p.row_scale,
                                p.dz,
                                static_cast<float*>(p.dz_lo),
                                static_cast<float*>(p.dzt_hi),
                                static_cast<float*>(p.dzt_lo),
                                p.ldz,
                                p.ldt,
                                p.T,
                                p.slab0,
                                p.slab_w};
  return run_gemm<true, DzEpi<true>>(tx_hi, tw_hi, tx_lo, tw_lo, p.T, p.slab_w, p.H, p.status,
                                     p.sms, p.stream, ea, true, FLCE_ROLE_DZ);
}

// grad_W (A = dz slab, B = x, both MN-major, K = T) and grad_x (A = dz slab K-major, B = W slab
// MN-major, K = slab width) of one slab in a single launch: both read only the dz slab written
// by the preceding dz launch, and one combined tile list fills the GPU evenly (two separate
// launches would each end in a partly filled last wave). The problem with the longer K (the
// longer tiles) is listed first, so that the tiles handed out last are the short ones.
cudaError_t launch_grads_bf16(const CUtensorMap& tdz_mn, const CUtensorMap& tx_mn,
                              const CUtensorMap& tdz_k, const CUtensorMap& tw_mn,
                              const GradWLaunch& pw, const GradXLaunch& px) {
  typename GradWEpi<false>::Args ew{pw.grad_w, pw.grad_loss, pw.scale, pw.H, pw.slab0, pw.slab_w};
  typename GradXEpi<false>::Args ex{px.acc,   px.grad_x, px.grad_loss, px.scale,
                                    px.T,     px.H,      px.mode};
  const Core core = role_core(pw.sms, FLCE_ROLE_GRADS);  // dz K-major map boxed to match
  const int rows = core_tile_rows(core);
  const GemmProblem w = make_problem(pw.slab_w, pw.H, pw.T, 64, true, true, rows, 0);
  const GemmProblem x = make_problem(px.T, px.H, px.K, 64, false, true, rows, 0);
  GemmGrid g{};
  g.num_problems = 2;
  g.status = pw.status;
  g.tile_counter = pw.tile_counter;
  if (x.k_blocks > w.k_blocks) {  // grad_x tiles first
    g.p[0] = x;
    g.p[1] = w;
    g.p[1].tile_begin = x.m_tiles * x.n_tiles;
    if (core != kCoreSingle)
      return launch_pair_core<GradXEpi<false>, GradWEpi<false>>(core, tdz_k, tw_mn, tdz_mn, tx_mn,
                                                                g, ex, ew, pw.sms, pw.stream,
                                                                FLCE_ROLE_GRADS);
    return launch_gemm<false, GradXEpi<false>, GradWEpi<false>>(tdz_k, tw_mn, tdz_mn, tx_mn, g, ex,
                                                                ew, pw.sms, pw.stream);
  }
  g.p[0] = w;
  g.p[1] = x;
  g.p[1].tile_begin = w.m_tiles * w.n_tiles;
  if (core != kCoreSingle)
    return launch_pair_core<GradWEpi<false>, GradXEpi<false>>(core, tdz_mn, tx_mn, tdz_k, tw_mn, g,
                                                              ew, ex, pw.sms, pw.stream,
                                                              FLCE_ROLE_GRADS);
  return launch_gemm<false, GradWEpi<false>, GradXEpi<false>>(tdz_mn, tx_mn, tdz_k, tw_mn, g, ew,
                                                              ex, pw.sms, pw.stream);
}

int pair_roles(int sms) {
  const int t = tune_sm_pairs();
  if (t >= 0) return t;
  // Automatic choice, decided once per device: all roles on pairs when every SM can hold half
  // of a resident pair of the kernel the automatic choice launches (wide tiles).
  static std::atomic<int> decided[64];  // 0: not yet; else mask + 1
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) {
    const int d = decided[dev].load();
    if (d) return d - 1;
  }
  auto kern = k_umma_gemm_pair<256, 1, GradXEpi<false>, GradWEpi<false>>;
  int mask = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairGeom<256, 1>::kSmemBytes) == cudaSuccess)
    mask = 2 * pair_resident_clusters<256, 1>(kern, sms) >= 2 * (sms / 2) ? kAutoPairRoles : 0;
  else
    cudaGetLastError();
  if (dev >= 0 && dev < 64) decided[dev].store(mask + 1);
  return mask;
}

cudaError_t launch_gradw_tf32(const CUtensorMap& tdzt_hi, const CUtensorMap& txt_hi,
                              const CUtensorMap& tdzt_lo, const CUtensorMap& txt_lo,
                              const GradWLaunch& p) {
  typename GradWEpi<true>::Args ea{p.grad_w, p.grad_loss, p.scale, p.H, p.slab0, p.slab_w};
  return run_gemm<true, GradWEpi<true>>(tdzt_hi, txt_hi, tdzt_lo, txt_lo, p.slab_w, p.H, p.T,
                                        p.status, p.sms, p.stream, ea, false, FLCE_ROLE_GRADS);
}

cudaError_t launch_gradx_tf32(const CUtensorMap& tdz_hi, const CUtensorMap& twt_hi,
                              const CUtensorMap& tdz_lo, const CUtensorMap& twt_lo,
                              const GradXLaunch& p) {
  typename GradXEpi<true>::Args ea{p.acc, p.grad_x, p.grad_loss, p.scale, p.T, p.H, p.mode};
  return run_gemm<true, GradXEpi<true>>(tdz_hi, twt_hi, tdz_lo, twt_lo, p.T, p.H, p.K, p.status,
                                        p.sms, p.stream, ea, false, FLCE_ROLE_GRADS);
}

// ---------------------------------------------------------------------------- TF32 split
// hi = x rounded to TF32 (10 mantissa bits, nearest), lo = x - hi (exact). Without `transpose`
// the outputs are [rows][ld_out]; with it they are [cols][ld_out] (ld_out >= rows). A 32 x 32
// shared tile keeps both the loads and the transposed stores coalesced.
__global__ void __launch_bounds__(256)
    k_split_tf32(const float* __restrict__ src, int64_t rows, int64_t cols, int64_t ld_out,
                 float* __restrict__ hi, float* __restrict__ lo, int transpose) {
  __shared__ float th[32][33];
  __shared__ float tl[32][33];
  const int64_t row_tiles = (rows + 31) / 32;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  for (int64_t rt = blockIdx.y; rt < row_tiles; rt += gridDim.y) {
    const int64_t r0 = rt * 32;
    for (int i = ty; i < 32; i += 8) {
      const int64_t r = r0 + i, c = c0 + tx;
      float h = 0.f, l = 0.f;
      if (r < rows && c < cols) split_tf32(src[r * cols + c], h, l);
      if (!transpose) {
        if (r < rows && c < cols) {
          hi[r * ld_out + c] = h;
          lo[r * ld_out + c] = l;
        }
      } else {
        th[i][tx] = h;
        tl[i][tx] = l;
      }
    }
    if (!transpose) continue;
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
      const int64_t c = c0 + i, r = r0 + tx;  // output row c, column r
      if (c < cols && r < rows) {
        hi[c * ld_out + r] = th[tx][i];
        lo[c * ld_out + r] = tl[tx][i];
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_split_tf32(const float* src, int64_t rows, int64_t cols, int64_t ld_out,
                              float* hi, float* lo, bool transpose, cudaStream_t stream) {
  const int64_t row_tiles = (rows + 31) / 32;
  dim3 grid(static_cast<unsigned>((cols + 31) / 32),
            static_cast<unsigned>(row_tiles < 65535 ? row_tiles : 65535));
  k_split_tf32<<<grid, 256, 0, stream>>>(src, rows, cols, ld_out, hi, lo, transpose ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace flce
