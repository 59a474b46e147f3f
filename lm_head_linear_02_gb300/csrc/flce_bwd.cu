// flce_bwd.cu - backward kernels, one vocab slab [slab0, slab0 + slab_w) at a time:
//   dz     : recompute z = x . W_slab^T and form dz = (softmax - onehot) * g  (slab buffer)
//   grad_W : grad_W[slab] = dz_slab^T . x                                     (K = T, complete)
//   grad_x : grad_x (+)= dz_slab . W_slab                                     (split-K over slabs)
// plus the TF32 hi/lo operand split used by the fp32 path.
#include "epilogues.cuh"
#include "flce_internal.h"

namespace flce {

template <bool kAMn, bool kBMn, bool kTF32, class Epi>
static cudaError_t run_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ta_lo,
                            const CUtensorMap& tb_lo, int M, int N, int K, int* status, int sms,
                            cudaStream_t stream, const typename Epi::Args& ea) {
  using G = StageGeom<kTF32>;
  auto kern = k_umma_gemm<kAMn, kBMn, kTF32, Epi>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes);
  if (e != cudaSuccess) return e;
  GemmGrid g;
  g.m_tiles = (M + kBM - 1) / kBM;
  g.n_tiles = (N + kBN - 1) / kBN;
  g.k_blocks = (K + G::kBK - 1) / G::kBK;
  g.group_m = kGroupM;
  g.status = status;
  const int tiles = g.m_tiles * g.n_tiles;
  const int grid = tiles < sms ? tiles : sms;
  kern<<<grid, kThreads, G::kSmemBytes, stream>>>(ta, tb, ta_lo, tb_lo, g, ea);
  return cudaGetLastError();
}

cudaError_t launch_dz_bf16(const CUtensorMap& tx, const CUtensorMap& tw_slab, const DzLaunch& p) {
  typename DzEpi<false>::Args ea{p.target, p.lse, p.dz, nullptr, nullptr, nullptr,
                                 p.ldz,    p.ldt, p.T,  p.slab0, p.slab_w};
  return run_gemm<false, false, false, DzEpi<false>>(tx, tw_slab, tx, tw_slab, p.T, p.slab_w, p.H,
                                                     p.status, p.sms, p.stream, ea);
}

cudaError_t launch_dz_tf32(const CUtensorMap& tx_hi, const CUtensorMap& tw_hi,
                           const CUtensorMap& tx_lo, const CUtensorMap& tw_lo, const DzLaunch& p) {
  typename DzEpi<true>::Args ea{p.target,
                                p.lse,
                                p.dz,
                                static_cast<float*>(p.dz_lo),
                                static_cast<float*>(p.dzt_hi),
                                static_cast<float*>(p.dzt_lo),
                                p.ldz,
                                p.ldt,
                                p.T,
                                p.slab0,
                                p.slab_w};
  return run_gemm<false, false, true, DzEpi<true>>(tx_hi, tw_hi, tx_lo, tw_lo, p.T, p.slab_w, p.H,
                                                   p.status, p.sms, p.stream, ea);
}

cudaError_t launch_gradw_bf16(const CUtensorMap& tdz_mn, const CUtensorMap& tx_mn,
                              const GradWLaunch& p) {
  typename GradWEpi<false>::Args ea{p.grad_w, p.grad_loss, p.scale, p.H, p.slab0, p.slab_w};
  return run_gemm<true, true, false, GradWEpi<false>>(tdz_mn, tx_mn, tdz_mn, tx_mn, p.slab_w, p.H,
                                                      p.T, p.status, p.sms, p.stream, ea);
}

cudaError_t launch_gradw_tf32(const CUtensorMap& tdzt_hi, const CUtensorMap& txt_hi,
                              const CUtensorMap& tdzt_lo, const CUtensorMap& txt_lo,
                              const GradWLaunch& p) {
  typename GradWEpi<true>::Args ea{p.grad_w, p.grad_loss, p.scale, p.H, p.slab0, p.slab_w};
  return run_gemm<false, false, true, GradWEpi<true>>(tdzt_hi, txt_hi, tdzt_lo, txt_lo, p.slab_w,
                                                      p.H, p.T, p.status, p.sms, p.stream, ea);
}

cudaError_t launch_gradx_bf16(const CUtensorMap& tdz_k, const CUtensorMap& tw_mn,
                              const GradXLaunch& p) {
  typename GradXEpi<false>::Args ea{p.acc, p.grad_x, p.grad_loss, p.scale, p.T, p.H, p.mode};
  return run_gemm<false, true, false, GradXEpi<false>>(tdz_k, tw_mn, tdz_k, tw_mn, p.T, p.H, p.K,
                                                       p.status, p.sms, p.stream, ea);
}

cudaError_t launch_gradx_tf32(const CUtensorMap& tdz_hi, const CUtensorMap& twt_hi,
                              const CUtensorMap& tdz_lo, const CUtensorMap& twt_lo,
                              const GradXLaunch& p) {
  typename GradXEpi<true>::Args ea{p.acc, p.grad_x, p.grad_loss, p.scale, p.T, p.H, p.mode};
  return run_gemm<false, false, true, GradXEpi<true>>(tdz_hi, twt_hi, tdz_lo, twt_lo, p.T, p.H,
                                                      p.K, p.status, p.sms, p.stream, ea);
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
