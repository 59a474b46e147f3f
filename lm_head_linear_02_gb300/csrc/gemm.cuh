// gemm.cuh - the single-SM warp-specialised tcgen05 contraction core, and what it shares with
// the CTA-pair core of gemm_pair.cuh: the problem and tile description (two problems per
// launch, raster groups, fixed-stride or counter-driven tile order), the tile queue depth, the
// per-warp store staging size and the host launch helpers.
//
// One CTA per SM, persistent over output tiles of BM x BN = 128 x 256 (one tcgen05.mma shape,
// M = 128 rows in the 128 TMEM lanes, N = 256 fp32 columns). Six warps:
//   warp 0      : TMA producer  - one thread streams K-slices of A and B into a kStages-deep
//                                 ring of 128B-swizzled shared-memory stages (mbarrier full/empty)
//   warp 1      : MMA issuer    - one thread issues tcgen05.mma into one of two TMEM
//                                 accumulators (2 x 256 columns) and commits to mbarriers
//   warps 2..5  : epilogue      - 128 threads, one accumulator row (TMEM lane) each, drain the
//                                 accumulator of tile j while the MMAs of tile j+1 run; each
//                                 warp owns kEpiStageBytes of shared memory after the ring for
//                                 transposing its global stores into coalesced ones
// The contraction itself (D = A . B^T over K) is all this file knows; what happens to a
// finished tile (online log-sum-exp, dz formation, gradient stores) is the Epi policy.
//
// Operand majors: A is [M][K] (K-major) or [K][M] (MN-major), B is [N][K] or [K][N]. MN-major
// is used for the backward contractions whose reduction runs over tokens or vocab rows.
// For fp32 inputs (kTF32x3) each operand arrives as a (hi, lo) pair of TF32-exact copies and
// each K-step issues hi.hi + hi.lo + lo.hi, which carries ~fp32 accuracy on TF32 tensor cores.
// The tensor core's additions into an fp32 accumulator do not round to nearest (their errors
// all lean one way) and the error of each is a fraction of the accumulator's last place, so
// the large hi.hi products and the small correction products go to separate accumulators (the
// two 256-column halves of TMEM; no double buffering on this path) and the epilogue adds the
// two in fp32: the large accumulator sees a third of the additions, the small one has tiny
// last places.
#pragma once

#include "flce_internal.h"
#include "ptx.cuh"

namespace flce {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kThreads = 192;
// Shared memory each epilogue warp owns for transposing its stores (32 rows x 64 bytes).
constexpr uint32_t kEpiStageBytes = 2048;
constexpr int kEpiWarp0 = 2;
constexpr uint32_t kTmemCols = 512;  // all of TMEM: two 256-column fp32 accumulators, or one
                                     // accumulator of two 256-column halves (wide pair tiles)

// One contraction D[M][N] = A . B^T of a launch. A launch carries one or two problems; their
// tiles form one list (problem 0 first) that the persistent CTAs walk with a fixed stride or,
// with a tile counter, take in list order as they become free.
struct GemmProblem {
  int m_tiles;     // ceil(M / tile rows)
  int n_tiles;     // ceil(N / 256)
  int k_blocks;    // ceil(K / BK)
  int a_mn, b_mn;  // operand majors (1 = MN-major; bf16 only)
  int group_m;     // raster: tiles walk N inside groups of group_m consecutive M tiles ...
  int group_n;     // ... or, when group_n > 0, walk M inside groups of group_n N tiles
  int tile_begin;  // first linear tile of this problem within the launch
};

struct GemmGrid {
  GemmProblem p[2];
  int num_problems;
  int num_tiles;
  int* status;        // device status word (FLCE_STATUS_* bits)
  int* tile_counter;  // null: CTA b takes tiles b, b + grid, ...; else a zeroed device int that
                      // hands out tiles in list order to whichever CTA is free (dynamic)
  int withhold;       // testing aid: CTA 0 (pair 0) does not signal its first accumulator tile
  int ordered;        // wide pair tiles only: drain the two 128-row halves one after the other
                      // (see k_umma_gemm_pair); 0 on every other core
};

// Depth of the per-CTA queue through which the producer hands tile indices to the MMA thread
// and the epilogue warps.
constexpr int kTileQueue = 4;

// The fields of the problem a tile belongs to, selected field by field (no dynamic indexing of
// the parameter array, so everything stays in registers).
struct TileInfo {
  int prob, mb, nb, k_blocks, a_mn, b_mn;
};

__device__ __forceinline__ TileInfo map_tile(const GemmGrid& g, int t) {
  const bool second = g.num_problems > 1 && t >= g.p[1].tile_begin;
  const int m_tiles = second ? g.p[1].m_tiles : g.p[0].m_tiles;
  const int n_tiles = second ? g.p[1].n_tiles : g.p[0].n_tiles;
  const int group_m = second ? g.p[1].group_m : g.p[0].group_m;
  const int group_n = second ? g.p[1].group_n : g.p[0].group_n;
  const int r = t - (second ? g.p[1].tile_begin : g.p[0].tile_begin);
  TileInfo ti;
  ti.prob = second ? 1 : 0;
  if (group_n > 0) {
    // groups of group_n consecutive N tiles (their B rows stay in L2); A streams past them,
    // every N tile of the group taken for one M tile before the next M tile
    const int per_group = group_n * m_tiles;
    const int grp = r / per_group;
    const int first = grp * group_n;
    const int gsz = min(group_n, n_tiles - first);
    const int q = r - grp * per_group;
    ti.mb = q / gsz;
    ti.nb = first + q % gsz;
  } else {
    const int per_group = group_m * n_tiles;
    const int grp = r / per_group;
    const int first = grp * group_m;
    const int gsz = min(group_m, m_tiles - first);
    const int q = r - grp * per_group;
    ti.mb = first + q % gsz;
    ti.nb = q / gsz;
  }
  ti.k_blocks = second ? g.p[1].k_blocks : g.p[0].k_blocks;
  ti.a_mn = second ? g.p[1].a_mn : g.p[0].a_mn;
  ti.b_mn = second ? g.p[1].b_mn : g.p[0].b_mn;
  return ti;
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
  // ring, barrier/slot block (1 KB), 2 KB of store staging per epilogue warp, alignment slack
  static constexpr uint32_t kSmemBytes = kRingBytes + 1024 + 4 * kEpiStageBytes + 1024;
};

// What an epilogue warp is given for one finished tile (one 128-row block of accumulators).
// Its 32 threads own one row each (one TMEM lane) and drain the 32-column chunks
// [c_begin, c_end) of the block's 256 columns. With split = 2 two warps share the same rows and
// take the column halves (part 0: chunks 0-3, part 1: chunks 4-7). An epilogue that needs
// per-row results of both halves passes them from part 1 to part 0 through xchg (two sets of
// 32 float4 slots, alternating with `iter`, the warp's tile count) and the mbarrier xbar (32
// arrivals per tile, phase parity iter & 1): part 1 writes and arrives, part 0 waits, bounded
// like every pipeline wait, so a partner that left on the abort path cannot hang it.
// Per-row inputs of an epilogue (target id, log-sum-exp, upstream factor of this thread's row),
// loaded by Epi::fetch as soon as the tile index is known, while the accumulator is still being
// computed, so that their global-memory latency is not paid after the tile is finished.
struct EpiRows {
  long long y;
  float lse;
  float scale;
};

struct EpiCtx {
  int row;            // accumulator row of this thread within the 128-row block
  uint32_t taddr;     // TMEM address of this warp's lane quarter, column 0 of the block
  uint4* stage;       // this warp's kEpiStageBytes of store staging
  int c_begin, c_end; // 32-column chunks of the block this warp drains
  int part, split;    // column half (0 / 1) and warps per row block (1 / 2)
  int iter;           // tiles this warp has drained before this one
  int two_acc;        // 1: the tile is the sum of two accumulators, taddr and taddr_corr
  uint32_t taddr_corr;
  uint32_t xbar;      // exchange mbarrier of the two warps sharing rows (split 2)
  float4* xchg;       // exchange slots of those two warps (split 2)
  int* status;        // device status word (a timed-out exchange sets FLCE_STATUS_TIMEOUT)
  volatile int* abort;
  EpiRows rows;       // this row's inputs (Epi::fetch with the same 128-row block index)
};

struct NoEpi {
  struct Args {};
  struct State {};
  static __device__ __forceinline__ void init(const Args&, State&) {}
  static __device__ __forceinline__ void fetch(const Args&, int, int, EpiRows&) {}
  static __device__ __forceinline__ void tile(const Args&, State&, int, int, const EpiCtx&) {}
};

// A stage holds [A_hi][A_lo][B_hi][B_lo] (lo copies only for kTF32x3, whose operands are
// K-major and whose launches carry one problem: tA0/tB0 hold hi, tA1/tB1 hold lo).
template <bool kTF32x3, class Epi0, class Epi1>
__global__ void __launch_bounds__(kThreads, 1)
    k_umma_gemm(const __grid_constant__ CUtensorMap tA0, const __grid_constant__ CUtensorMap tB0,
                const __grid_constant__ CUtensorMap tA1, const __grid_constant__ CUtensorMap tB1,
                const GemmGrid g, const typename Epi0::Args e0, const typename Epi1::Args e1) {
  using G = StageGeom<kTF32x3>;
  constexpr uint32_t kFmt = kTF32x3 ? kFmtTF32 : kFmtBF16;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kRingBytes);
  // bars[0..S) full, [S..2S) empty, [2S..2S+2) tmem_full, [2S+2..2S+4) tmem_empty, [2S+4] drain,
  // [2S+5..2S+5+Q) tile-queue full, [2S+5+Q..2S+5+2Q) tile-queue empty
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * G::kStages + 5 + 2 * kTileQueue);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // Pipeline counters kept in shared memory so that an aborted CTA can wait out its own
  // copies and MMAs still in flight before it frees TMEM and exits.
  int* issued_fills = reinterpret_cast<int*>(tmem_slot + 2);
  int* consumed_fills = reinterpret_cast<int*>(tmem_slot + 3);
  volatile int* tile_q = reinterpret_cast<volatile int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (G::kStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * G::kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * G::kStages + 2 + a); };
  auto drain_bar = [&]() { return bar0 + 8u * (2 * G::kStages + 4); };
  auto tq_full = [&](int q) { return bar0 + 8u * (2 * G::kStages + 5 + q); };
  auto tq_empty = [&](int q) { return bar0 + 8u * (2 * G::kStages + 5 + kTileQueue + q); };

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
    for (int q = 0; q < kTileQueue; ++q) {
      mbar_init(tq_full(q), 1);   // the producer publishes a tile index
      mbar_init(tq_empty(q), 5);  // the MMA thread and the 4 epilogue warps have read it
    }
    *abort_flag = 0;
    *issued_fills = 0;
    *consumed_fills = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tA0);
    tma_prefetch(&tB0);
    if (kTF32x3 || g.num_problems > 1) {
      tma_prefetch(&tA1);
      tma_prefetch(&tB1);
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

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fills = 0;
      bool ok = true;
      int qslot = 0;
      uint32_t qphase = 0;
      for (int i = 0; ok; ++i) {
        // Next tile (static stride or the shared counter); -1 ends the queue for the consumers.
        int t = g.tile_counter ? atomicAdd(g.tile_counter, 1)
                               : static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
        if (t >= g.num_tiles) t = -1;
        if (!mbar_wait(tq_empty(qslot), qphase ^ 1u, g.status, abort_flag)) break;
        tile_q[qslot] = t;
        mbar_arrive(tq_full(qslot));
        if (++qslot == kTileQueue) {
          qslot = 0;
          qphase ^= 1u;
        }
        if (t < 0) break;
        const TileInfo ti = map_tile(g, t);
        const CUtensorMap* ta = (!kTF32x3 && ti.prob) ? &tA1 : &tA0;
        const CUtensorMap* tb = (!kTF32x3 && ti.prob) ? &tB1 : &tB0;
        const int m0 = ti.mb * kBM, n0 = ti.nb * kBN;
        const bool a_mn = !kTF32x3 && ti.a_mn != 0;
        const bool b_mn = !kTF32x3 && ti.b_mn != 0;
        const int k_blocks = ti.k_blocks;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, g.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, G::kStageBytes);
          const uint32_t sA = ring + stage * G::kStageBytes;
          const uint32_t sB = sA + G::kCopies * G::kABytes;
          const int k0 = kb * G::kBK;
          if (!a_mn) {
            tma_load_2d(sA, ta, fb, k0, m0);
            if constexpr (kTF32x3) tma_load_2d(sA + G::kABytes, &tA1, fb, k0, m0);
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j) tma_load_2d(sA + j * 8192u, ta, fb, m0 + 64 * j, k0);
          }
          if (!b_mn) {
            tma_load_2d(sB, tb, fb, k0, n0);
            if constexpr (kTF32x3) tma_load_2d(sB + G::kBBytes, &tB1, fb, k0, n0);
          } else {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j) tma_load_2d(sB + j * 8192u, tb, fb, n0 + 64 * j, k0);
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
      int qslot = 0;
      uint32_t qphase = 0;
      while (ok) {
        if (!mbar_wait(tq_full(qslot), qphase, g.status, abort_flag)) break;
        const int t = tile_q[qslot];
        mbar_arrive(tq_empty(qslot));
        if (++qslot == kTileQueue) {
          qslot = 0;
          qphase ^= 1u;
        }
        if (t < 0) break;
        const TileInfo ti = map_tile(g, t);
        const bool a_mn = !kTF32x3 && ti.a_mn != 0;
        const bool b_mn = !kTF32x3 && ti.b_mn != 0;
        const int k_blocks = ti.k_blocks;
        const uint32_t idesc = idesc_f32acc(kFmt, kBM, kBN, a_mn, b_mn);
        // Stage-0 descriptors and the per-K-step advance (16-byte units): K-major moves 32 B
        // along the swizzled row, MN-major moves 16 bf16 K rows of 128 B.
        const uint32_t sB0 = ring + G::kCopies * G::kABytes;
        const uint64_t a_base =
            a_mn ? sdesc_sw128(ring, 8192u, 1024u) : sdesc_sw128(ring, 16u, 1024u);
        const uint64_t b_base =
            b_mn ? sdesc_sw128(sB0, 8192u, 1024u) : sdesc_sw128(sB0, 16u, 1024u);
        const uint64_t a_step = a_mn ? (2048u >> 4) : (32u >> 4);
        const uint64_t b_step = b_mn ? (2048u >> 4) : (32u >> 4);
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, g.status, abort_flag)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        const uint32_t d_corr = tmem_base + static_cast<uint32_t>(kBN);  // kTF32x3: corrections
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, g.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t soff = static_cast<uint64_t>(stage * G::kStageBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a_hi = a_base + soff + kk * a_step;
            const uint64_t b_hi = b_base + soff + kk * b_step;
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if constexpr (!kTF32x3) {
              mma_bf16(d_tmem, a_hi, b_hi, idesc, accum);
            } else {
              const uint64_t a_lo = a_hi + (G::kABytes >> 4);
              const uint64_t b_lo = b_hi + (G::kBBytes >> 4);
              mma_tf32(d_corr, a_lo, b_hi, idesc, accum);
              mma_tf32(d_corr, a_hi, b_lo, idesc, 1u);
              mma_tf32(d_tmem, a_hi, b_hi, idesc, accum);
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
        // (g.withhold: the failure-path test leaves CTA 0's first tile unsignalled so that its
        // epilogue's bounded wait runs out.)
        if (!(g.withhold && blockIdx.x == 0 && consumed == k_blocks)) mma_commit(tfull_bar(acc));
        if (kTF32x3) {  // one (two-part) accumulator
          acc_phase ^= 1u;
        } else if (++acc == 2) {
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
    uint4* stage = reinterpret_cast<uint4*>(smem + G::kRingBytes + 1024 +
                                            static_cast<uint32_t>(warp - 2) * kEpiStageBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    typename Epi0::State st0;
    typename Epi1::State st1;
    Epi0::init(e0, st0);
    Epi1::init(e1, st1);
    int qslot = 0;
    uint32_t qphase = 0;
    while (true) {
      if (!mbar_wait(tq_full(qslot), qphase, g.status, abort_flag)) break;
      const int t = tile_q[qslot];
      __syncwarp();
      if (lane == 0) mbar_arrive(tq_empty(qslot));
      if (++qslot == kTileQueue) {
        qslot = 0;
        qphase ^= 1u;
      }
      if (t < 0) break;
      const TileInfo ti = map_tile(g, t);
      EpiRows rows;
      if (ti.prob == 0)
        Epi0::fetch(e0, ti.mb, row, rows);
      else
        Epi1::fetch(e1, ti.mb, row, rows);
      if (!mbar_wait(tfull_bar(acc), acc_phase, g.status, abort_flag)) break;
      tc_fence_after_sync();
      __syncwarp();
      EpiCtx ctx;
      ctx.row = row;
      ctx.taddr =
          tmem_base + static_cast<uint32_t>(acc * kBN) + (static_cast<uint32_t>(quarter * 32) << 16);
      ctx.stage = stage;
      ctx.c_begin = 0;
      ctx.c_end = kBN / 32;
      ctx.part = 0;
      ctx.split = 1;
      ctx.iter = 0;
      ctx.two_acc = kTF32x3 ? 1 : 0;
      ctx.taddr_corr = ctx.taddr + static_cast<uint32_t>(kBN);
      ctx.xbar = 0;
      ctx.xchg = nullptr;
      ctx.status = g.status;
      ctx.abort = abort_flag;
      ctx.rows = rows;
      if (ti.prob == 0)
        Epi0::tile(e0, st0, ti.mb, ti.nb, ctx);
      else
        Epi1::tile(e1, st1, ti.mb, ti.nb, ctx);
      tc_fence_before_sync();
      mbar_arrive(tempty_bar(acc));
      if (kTF32x3) {
        acc_phase ^= 1u;
      } else if (++acc == 2) {
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

// ---------------------------------------------------------------------------- host helpers

// Problem description for a launch; `tile_rows` is 128 for this core, 256 or 512 for CTA
// pairs. `vocab_n`: the N dimension is the vocabulary (B = weight rows), which is rastered in
// groups of tune_raster_vocab() rows when that is set, instead of groups of M rows.
inline GemmProblem make_problem(int M, int N, int K, int bk, bool a_mn, bool b_mn, int tile_rows,
                                int tile_begin, bool vocab_n = false) {
  GemmProblem p;
  p.m_tiles = (M + tile_rows - 1) / tile_rows;
  p.n_tiles = (N + kBN - 1) / kBN;
  p.k_blocks = (K + bk - 1) / bk;
  p.a_mn = a_mn ? 1 : 0;
  p.b_mn = b_mn ? 1 : 0;
  const int g = tune_raster_rows() / tile_rows;
  p.group_m = g > 0 ? g : 1;
  p.group_n = vocab_n ? tune_raster_vocab() / kBN : 0;
  p.tile_begin = tile_begin;
  return p;
}

inline void finish_grid(GemmGrid& g) {
  g.num_tiles = 0;
  for (int i = 0; i < g.num_problems; ++i)
    g.num_tiles = g.p[i].tile_begin + g.p[i].m_tiles * g.p[i].n_tiles;
}

// Launch one or two problems on a persistent grid of single CTAs (one per SM, at most one
// per tile).
template <bool kTF32x3, class Epi0, class Epi1>
cudaError_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
                        const CUtensorMap& b1, GemmGrid g, const typename Epi0::Args& e0,
                        const typename Epi1::Args& e1, int sms, cudaStream_t stream) {
  using G = StageGeom<kTF32x3>;
  auto kern = k_umma_gemm<kTF32x3, Epi0, Epi1>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes);
  if (e != cudaSuccess) return e;
  finish_grid(g);
  if (g.tile_counter) {
    e = cudaMemsetAsync(g.tile_counter, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
  }
  g.withhold = take_withhold_request() ? 1 : 0;
  const int grid = g.num_tiles < sms ? g.num_tiles : sms;
  kern<<<grid, kThreads, G::kSmemBytes, stream>>>(a0, b0, a1, b1, g, e0, e1);
  return cudaGetLastError();
}

}  // namespace flce
