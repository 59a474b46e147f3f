// gemm.cuh - the warp-specialised tcgen05 contraction core shared by every FLCE kernel.
//
// One CTA per SM, persistent over output tiles of BM x BN = 128 x 256 (one tcgen05.mma shape,
// M = 128 rows in the 128 TMEM lanes, N = 256 fp32 columns). Six warps:
//   warp 0      : TMA producer  - one thread streams K-slices of A and B into a kStages-deep
//                                 ring of 128B-swizzled shared-memory stages (mbarrier full/empty)
//   warp 1      : MMA issuer    - one thread issues tcgen05.mma into one of two TMEM
//                                 accumulators (2 x 256 columns) and commits to mbarriers
//   warps 2..5  : epilogue      - 128 threads, one accumulator row (TMEM lane) each, drain the
//                                 accumulator of tile j while the MMAs of tile j+1 run
// The contraction itself (D = A . B^T over K) is all this file knows; what happens to a
// finished tile (online log-sum-exp, dz formation, gradient stores) is the Epi policy.
//
// Operand majors: A is [M][K] (K-major) or [K][M] (MN-major), B is [N][K] or [K][N]. MN-major
// is used for the backward contractions whose reduction runs over tokens or vocab rows.
// For fp32 inputs (kTF32x3) each operand arrives as a (hi, lo) pair of TF32-exact copies and
// each K-step issues hi.hi + hi.lo + lo.hi, which carries ~fp32 accuracy on TF32 tensor cores.
#pragma once

#include "ptx.cuh"

namespace flce {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kThreads = 192;
constexpr int kEpiWarp0 = 2;
constexpr uint32_t kTmemCols = 512;  // two 256-column fp32 accumulators

struct GemmGrid {
  int m_tiles;   // ceil(M / 128)
  int n_tiles;   // ceil(N / 256)
  int k_blocks;  // ceil(K / BK)
  int group_m;   // raster: tiles walk N inside groups of group_m consecutive M tiles
  int* status;   // device status word (FLCE_STATUS_* bits)
};

__device__ __forceinline__ void map_tile(const GemmGrid& g, int t, int& mb, int& nb) {
  const int per_group = g.group_m * g.n_tiles;
  const int grp = t / per_group;
  const int first = grp * g.group_m;
  const int gsz = min(g.group_m, g.m_tiles - first);
  const int r = t - grp * per_group;
  mb = first + r % gsz;
  nb = r / gsz;
}

template <bool kTF32x3>
struct StageGeom {
  static constexpr int kElem = kTF32x3 ? 4 : 2;
  static constexpr int kBK = 128 / kElem;                    // one 128-byte swizzle row of K
  static constexpr uint32_t kABytes = kBM * 128;             // 16 KB per operand copy
  static constexpr uint32_t kBBytes = kBN * 128;             // 32 KB per operand copy
  static constexpr int kCopies = kTF32x3 ? 2 : 1;            // hi (+ lo)
  static constexpr uint32_t kStageBytes = kCopies * (kABytes + kBBytes);
  static constexpr int kStages = kTF32x3 ? 2 : 4;
  static constexpr uint32_t kRingBytes = kStages * kStageBytes;
  // ring + barriers/bookkeeping + 1 KB alignment slack
  static constexpr uint32_t kSmemBytes = kRingBytes + 1024 + 1024;
};

// A stage holds [A_hi][A_lo][B_hi][B_lo] (lo copies only for kTF32x3).
template <bool kAMn, bool kBMn, bool kTF32x3, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    k_umma_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmA_lo,
                const __grid_constant__ CUtensorMap tmB_lo, const GemmGrid g,
                const typename Epi::Args ea) {
  using G = StageGeom<kTF32x3>;
  static_assert(!(kTF32x3 && (kAMn || kBMn)), "TF32 operands are K-major only");
  constexpr uint32_t kIdesc = idesc_f32acc(kTF32x3 ? kFmtTF32 : kFmtBF16, kBM, kBN, kAMn, kBMn);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kRingBytes);
  // bars[0..S) full, [S..2S) empty, [2S..2S+2) tmem_full, [2S+2..2S+4) tmem_empty, [2S+4] drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * G::kStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (G::kStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * G::kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * G::kStages + 2 + a); };

  auto drain_bar = [&]() { return bar0 + 8u * (2 * G::kStages + 4); };
  // Pipeline counters kept in shared memory so that an aborted CTA can wait out its own
  // copies and MMAs still in flight before it frees TMEM and exits.
  int* issued_fills = reinterpret_cast<int*>(tmem_slot + 2);
  int* consumed_fills = reinterpret_cast<int*>(tmem_slot + 3);

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 128);
    }
    mbar_init(drain_bar(), 1);
    *abort_flag = 0;
    *issued_fills = 0;
    *consumed_fills = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
    if (kTF32x3) {
      tma_prefetch(&tmA_lo);
      tma_prefetch(&tmB_lo);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = g.m_tiles * g.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fills = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        map_tile(g, t, mb, nb);
        const int m0 = mb * kBM, n0 = nb * kBN;
        for (int kb = 0; kb < g.k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, g.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, G::kStageBytes);
          const uint32_t sA = ring + stage * G::kStageBytes;
          const uint32_t sB = sA + G::kCopies * G::kABytes;
          const int k0 = kb * G::kBK;
          if constexpr (!kAMn) {
            tma_load_2d(sA, &tmA, fb, k0, m0);
            if constexpr (kTF32x3) tma_load_2d(sA + G::kABytes, &tmA_lo, fb, k0, m0);
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j) tma_load_2d(sA + j * 8192u, &tmA, fb, m0 + 64 * j, k0);
          }
          if constexpr (!kBMn) {
            tma_load_2d(sB, &tmB, fb, k0, n0);
            if constexpr (kTF32x3) tma_load_2d(sB + G::kBBytes, &tmB_lo, fb, k0, n0);
          } else {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j) tma_load_2d(sB + j * 8192u, &tmB, fb, n0 + 64 * j, k0);
          }
          ++fills;
          if (++stage == G::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      *issued_fills = fills;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int consumed = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, g.status, abort_flag)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < g.k_blocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, g.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sA = ring + stage * G::kStageBytes;
          const uint32_t sB = sA + G::kCopies * G::kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // K-major: advance 32 B along the swizzled row; MN-major: advance 16 (bf16) K rows.
            const uint64_t a_hi = kAMn ? sdesc_sw128(sA + kk * 2048u, 8192u, 1024u)
                                       : sdesc_sw128(sA + kk * 32u, 16u, 1024u);
            const uint64_t b_hi = kBMn ? sdesc_sw128(sB + kk * 2048u, 8192u, 1024u)
                                       : sdesc_sw128(sB + kk * 32u, 16u, 1024u);
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if constexpr (!kTF32x3) {
              mma_bf16(d_tmem, a_hi, b_hi, kIdesc, accum);
            } else {
              const uint64_t a_lo = sdesc_sw128(sA + G::kABytes + kk * 32u, 16u, 1024u);
              const uint64_t b_lo = sdesc_sw128(sB + G::kBBytes + kk * 32u, 16u, 1024u);
              mma_tf32(d_tmem, a_lo, b_hi, kIdesc, accum);
              mma_tf32(d_tmem, a_hi, b_lo, kIdesc, 1u);
              mma_tf32(d_tmem, a_hi, b_hi, kIdesc, 1u);
            }
          }
          mma_commit(empty_bar(stage));
          ++consumed;
          if (++stage == G::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      *consumed_fills = consumed;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lane group this warp may access
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    typename Epi::State st;
    Epi::init(ea, st);
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      if (!mbar_wait(tfull_bar(acc), acc_phase, g.status, abort_flag)) break;
      tc_fence_after_sync();
      __syncwarp();
      int mb, nb;
      map_tile(g, t, mb, nb);
      const uint32_t taddr =
          tmem_base + static_cast<uint32_t>(acc * kBN) + (static_cast<uint32_t>(quarter * 32) << 16);
      Epi::tile(ea, st, mb, nb, row, taddr);
      tc_fence_before_sync();
      mbar_arrive(tempty_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    // Some wait ran out of time. Before TMEM is freed and the CTA exits, let the MMAs this CTA
    // issued finish (one more commit drains them all) and let every TMA fill that the MMA warp
    // never consumed land in shared memory. Both waits are bounded and ignore the abort flag.
    if (warp == 1 && lane == 0) {
      mma_commit(drain_bar());
      mbar_wait_bounded(drain_bar(), 0u);
    }
    if (warp == 0 && lane == 0) {
      const int issued = *issued_fills;
      for (int f = *consumed_fills; f < issued; ++f)
        mbar_wait_bounded(full_bar(f % G::kStages), static_cast<uint32_t>((f / G::kStages) & 1));
    }
    __syncwarp();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace flce
