// gemm_pair.cuh - the contraction core on CTA pairs (tcgen05 cta_group::2): bf16 operands, or
// fp32 operands as 3xTF32 (hi, lo) copies on 128-row CTA tiles (kTF32x3, see PairGeom).
//
// A cluster of two CTAs on two SMs computes one (2 kRows) x 256 output tile with one MMA stream:
// CTA r holds rows [kRows r, kRows r + kRows) of the A tile and rows [128r, 128r + 128) of the
// B tile (the N dimension), the pair's tensor cores exchange the B halves, and CTA r's TMEM
// receives its kRows rows of D across all 256 columns. Two geometries:
//   kRows = 128: 256 x 256 pair tiles; a 64-deep K slice costs 32 KB per CTA (16 KB of A, 16 KB
//                of B), six pipeline stages, two 256-column accumulators (the epilogue of one
//                tile overlaps the main loop of the next).
//   kRows = 256: 512 x 256 pair tiles; each K step issues two M=256 MMAs (the CTA's two 128-row
//                halves of A against the same B), so a K slice costs 48 KB per CTA for twice the
//                FLOPs: 48 instead of 64 bytes of shared-memory fill per 1024 FLOPs. On GB300 the
//                TMA fill rate of one SM, not the tensor core, bounds the 128-row geometry (about
//                40-50 B per SM clock measured, 64 needed), so this one keeps the tensor pipe
//                busy; the price is one accumulator filling all 512 TMEM columns, so the epilogue
//                of a tile is only partly hidden: with the ordered drain (g.ordered) the 8
//                epilogue warps read the first 128-row half, hand its columns back, and the next
//                tile's MMAs on that half run while they read the second.
//
// Roles (per CTA: 2 + 4 (kRows / 128) kSplit warps):
//   warp 0 (both CTAs)   TMA producer: loads this CTA's A rows and B half; completion is counted
//                        on the LEADER's full barrier, which the leader arms for both CTAs.
//   warp 1 (leader)      MMA issuer: waits for both CTAs' bytes, issues M=256 N=256 MMAs, and
//                        commits to the empty / tmem-full barriers of BOTH CTAs (multicast).
//   warp 1 (peer)        idle (takes part in the pair's TMEM allocation only).
//   warps 2.. (both)     epilogue: warp 2 + 4h + q drains TMEM lanes [32q', 32q' + 32) of half h
//                        (q' = warp % 4, the lane quarter a warp may access), then tells the
//                        leader (remote mbarrier arrive) that the accumulator is free. With
//                        kSplit = 2 a second set of warps (2 + 4 kHalves + ...) takes columns
//                        128-255 of the same rows and the first set columns 0-127. Ordered
//                        drain (wide tiles, kSplit = 1): warp 2 + 4p + q takes columns
//                        [128p, 128p + 128) of lane quarter q' in half 0, then in half 1, and
//                        releases each half on its own barrier (tmem_empty 0 and 1).
// Each epilogue warp loads its rows' inputs (Epi::fetch) as soon as it knows the next tile,
// before the accumulator is ready, and releases TMEM with a CTA-scope arrive, which does not
// wait for the tile's global stores to become visible to the cluster.
// A launch may carry two independent problems: grad_W and grad_x of one vocab slab run together,
// so that their tiles fill the GPU in one wave pattern instead of two.
#pragma once

#include "gemm.cuh"

namespace flce {

// kSplit: epilogue warps per (lane quarter, 128-row half): 1 drains all 256 columns of its
// rows, 2 gives each of two warps 128 of them (16 epilogue warps on wide tiles), which halves
// the time a finished tile keeps the single accumulator of the wide geometry busy.
// kTF32x3: fp32 operands as TF32 (hi, lo) copies (3xTF32, 128-row CTA tiles only): a stage
// holds [A_hi][A_lo][B_hi][B_lo], each a 128-byte row of 32 fp32 per operand row, and the
// 512 TMEM columns hold one tile's two accumulators, hi.hi at column 0 and the corrections
// hi.lo + lo.hi at column 256 (kept apart so that the small terms are not truncated against
// the large ones), summed in fp32 by the epilogue.
template <int kRows, int kSplit = 1, bool kTF32x3 = false>
struct PairGeom {
  static_assert(kRows == 128 || kRows == 256, "rows per CTA: 128 or 256");
  static_assert(kSplit == 1 || kSplit == 2, "epilogue warps per row block: 1 or 2");
  static_assert(!kTF32x3 || (kRows == 128 && kSplit == 1), "3xTF32: 128-row CTA tiles");
  static constexpr int kHalves = kRows / 128;          // M=256 MMAs per K step / epilogue halves
  static constexpr int kCopies = kTF32x3 ? 2 : 1;      // hi (+ lo) copy of each operand
  static constexpr int kStages = kTF32x3 ? 3 : (kRows == 128 ? 6 : 4);
  static constexpr uint32_t kABytes = kRows * 128;     // kRows rows x 128 B (64 bf16 / 32 fp32)
  static constexpr uint32_t kBBytes = 128 * 128;       // this CTA's 128 N rows x 128 B
  static constexpr uint32_t kStageBytes = kCopies * (kABytes + kBBytes);
  static constexpr uint32_t kRingBytes = kStages * kStageBytes;
  static constexpr int kAccBufs = kTF32x3 ? 1 : 2 / kHalves;  // tiles in the 512 TMEM columns
  static constexpr int kEpiWarps = 4 * kHalves * kSplit;
  // ring, barrier/slot block (1 KB), store staging per epilogue warp, alignment slack
  static constexpr uint32_t kSmemBytes = kRingBytes + 1024 + kEpiWarps * kEpiStageBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kTileRows = 2 * kRows;          // M rows of one pair tile
};
constexpr int kPairBK = 64;

// GemmProblem::m_tiles counts pair tiles of 2 kRows rows (make_problem with tile_rows =
// PairGeom<kRows>::kTileRows) and the epilogue receives 128-row block indices.
template <int kRows, int kSplit, class Epi0, class Epi1, bool kTF32x3 = false>
__global__ void __cluster_dims__(2, 1, 1)
    __launch_bounds__(PairGeom<kRows, kSplit, kTF32x3>::kThreads, 1)
    k_umma_gemm_pair(const __grid_constant__ CUtensorMap tA0,
                     const __grid_constant__ CUtensorMap tB0,
                     const __grid_constant__ CUtensorMap tA1,
                     const __grid_constant__ CUtensorMap tB1, const GemmGrid g,
                     const typename Epi0::Args e0, const typename Epi1::Args e1) {
  using G = PairGeom<kRows, kSplit, kTF32x3>;
  // wide tiles with one warp per (lane quarter, column half) may drain their halves in order
  constexpr bool kOrderable = G::kHalves == 2 && kSplit == 1;
  constexpr int kBK = kTF32x3 ? 32 : kPairBK;  // K elements per stage (one 128-byte row)
  constexpr int kPairStages = G::kStages;
  constexpr uint32_t kPairABytes = G::kABytes;
  constexpr uint32_t kPairStageBytes = G::kStageBytes;
  constexpr uint32_t kPairRingBytes = G::kRingBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPairRingBytes);
  // bars: [0,S) full, [S,2S) empty, [2S,2S+2) tmem_full, [2S+2,2S+4) tmem_empty, [2S+4] drain
  // [2S+5, 2S+5+Q) tile-queue full, [2S+5+Q, 2S+5+2Q) tile-queue empty (used in the leader),
  // [2S+5+2Q, 2S+5+2Q+8) epilogue exchange, one per (lane quarter, half) row block (split 2)
  constexpr int kXBars = 8;
  uint32_t* slots =
      reinterpret_cast<uint32_t*>(bars + 2 * kPairStages + 5 + 2 * kTileQueue + kXBars);
  uint32_t* tmem_slot = slots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slots + 1);
  int* issued_fills = reinterpret_cast<int*>(slots + 2);
  int* consumed_fills = reinterpret_cast<int*>(slots + 3);
  volatile int* tile_q = reinterpret_cast<volatile int*>(slots + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kPairStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kPairStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kPairStages + 2 + a); };
  auto drain_bar = [&]() { return bar0 + 8u * (2 * kPairStages + 4); };
  auto tq_full = [&](int q) { return bar0 + 8u * (2 * kPairStages + 5 + q); };
  auto tq_empty = [&](int q) { return bar0 + 8u * (2 * kPairStages + 5 + kTileQueue + q); };
  auto x_bar = [&](int i) { return bar0 + 8u * (2 * kPairStages + 5 + 2 * kTileQueue + i); };
  // Tile indices flow through a small queue in each CTA: the leader's producer takes the next
  // tile (fixed stride or the shared counter) and writes it into both CTAs' queues; the
  // leader's MMA thread, the peer's producer and the epilogue warps of both CTAs read it and
  // release the slot back to the leader (1 + 1 + 2 kEpiWarps arrivals).
  auto tq_release = [&](int q) {
    if (leader)
      mbar_arrive(tq_empty(q));
    else
      mbar_arrive_cluster(mapa_shared(tq_empty(q), 0));
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full_bar(s), 1);   // leader: its own expect_tx arrive (+ both CTAs' bytes)
      mbar_init(empty_bar(s), 1);  // one multicast commit from the leader's MMA thread
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * G::kEpiWarps);  // leader: every epilogue warp of both CTAs
    }
    mbar_init(drain_bar(), 1);
    for (int q = 0; q < kTileQueue; ++q) {
      mbar_init(tq_full(q), 1);
      mbar_init(tq_empty(q), 2 + 2 * G::kEpiWarps);
    }
    for (int i = 0; i < kXBars; ++i) mbar_init(x_bar(i), 32);  // every lane of part 1
    *abort_flag = 0;
    *issued_fills = 0;
    *consumed_fills = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tA0);
    tma_prefetch(&tB0);
    if (kTF32x3 || g.num_problems > 1) {  // the second problem's maps, or the lo copies' maps
      tma_prefetch(&tA1);
      tma_prefetch(&tB1);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // barrier inits and TMEM allocation visible to both CTAs
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const int cluster_id = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;

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
        int t;
        if (leader) {
          t = g.tile_counter ? atomicAdd(g.tile_counter, 1) : cluster_id + i * n_clusters;
          if (t >= g.num_tiles) t = -1;
          if (!mbar_wait_cluster(tq_empty(qslot), qphase ^ 1u, g.status, abort_flag)) break;
          tile_q[qslot] = t;
          st_shared_cluster(mapa_shared(smem_u32(const_cast<int*>(tile_q + qslot)), 1), t);
          mbar_arrive(tq_full(qslot));
          mbar_arrive_cluster(mapa_shared(tq_full(qslot), 1));
        } else {
          if (!mbar_wait_cluster(tq_full(qslot), qphase, g.status, abort_flag)) break;
          t = tile_q[qslot];
          tq_release(qslot);
        }
        if (++qslot == kTileQueue) {
          qslot = 0;
          qphase ^= 1u;
        }
        if (t < 0) break;
        const TileInfo pt = map_tile(g, t);
        const CUtensorMap* ta = pt.prob ? &tA1 : &tA0;
        const CUtensorMap* tb = pt.prob ? &tB1 : &tB0;
        const int m0 = pt.mb * G::kTileRows + static_cast<int>(rank) * kRows;
        const int n0 = pt.nb * 256 + static_cast<int>(rank) * 128;
        const bool a_mn = !kTF32x3 && pt.a_mn != 0, b_mn = !kTF32x3 && pt.b_mn != 0;
        const int k_blocks = pt.k_blocks;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, g.status, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * kPairStageBytes);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t sA = ring + stage * kPairStageBytes;
          const uint32_t sB = sA + G::kCopies * kPairABytes;
          const int k0 = kb * kBK;
          if constexpr (kTF32x3) {  // K-major hi and lo copies: tA0/tB0 hi, tA1/tB1 lo
            tma_load_2d_pair(sA, &tA0, fb, k0, m0);
            tma_load_2d_pair(sA + kPairABytes, &tA1, fb, k0, m0);
            tma_load_2d_pair(sB, &tB0, fb, k0, n0);
            tma_load_2d_pair(sB + G::kBBytes, &tB1, fb, k0, n0);
          } else if (!a_mn) {  // one box of kRows rows (the A map is boxed {64 x kRows})
            tma_load_2d_pair(sA, ta, fb, k0, m0);
          } else {  // kRows / 64 boxes of {64 (M) x 64 (K)}
#pragma unroll
            for (int j = 0; j < kRows / 64; ++j)
              tma_load_2d_pair(sA + 8192u * j, ta, fb, m0 + 64 * j, k0);
          }
          if constexpr (!kTF32x3) {
            if (!b_mn) {
              tma_load_2d_pair(sB, tb, fb, k0, n0);
            } else {
              tma_load_2d_pair(sB, tb, fb, n0, k0);
              tma_load_2d_pair(sB + 8192u, tb, fb, n0 + 64, k0);
            }
          }
          ++fills;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      *issued_fills = fills;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (leader)
    if (leader && lane == 0) {
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
        tq_release(qslot);
        if (++qslot == kTileQueue) {
          qslot = 0;
          qphase ^= 1u;
        }
        if (t < 0) break;
        const TileInfo pt = map_tile(g, t);
        const bool a_mn = !kTF32x3 && pt.a_mn != 0, b_mn = !kTF32x3 && pt.b_mn != 0;
        const int k_blocks = pt.k_blocks;
        const uint32_t idesc =
            idesc_f32acc(kTF32x3 ? kFmtTF32 : kFmtBF16, 256, 256, a_mn, b_mn);
        // Descriptor of stage 0 and the per-K-step advance (in 16-byte units): K-major moves
        // 32 B along the swizzled row, MN-major moves 16 K rows of 128 B.
        const uint64_t a_base =
            a_mn ? sdesc_sw128(ring, 8192u, 1024u) : sdesc_sw128(ring, 16u, 1024u);
        const uint32_t sB0 = ring + G::kCopies * kPairABytes;
        const uint64_t b_base =
            b_mn ? sdesc_sw128(sB0, 8192u, 1024u) : sdesc_sw128(sB0, 16u, 1024u);
        const uint64_t a_step = a_mn ? (2048u >> 4) : (32u >> 4);
        const uint64_t b_step = b_mn ? (2048u >> 4) : (32u >> 4);
        // Accumulator handshake with both CTAs' epilogues: cluster-scope acquire.
        if (!mbar_wait_cluster(tempty_bar(acc), acc_phase ^ 1u, g.status, abort_flag)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * G::kHalves * kBN);
        // The MMAs of one 128-row half over the 64-deep K slice in ring stage s.
        auto issue_half = [&](int s, int h, int kb) {
          const uint64_t soff = static_cast<uint64_t>(s * kPairStageBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // half h: A rows [128h, 128h + 128), +16 KB
            mma_bf16_pair(d_tmem + static_cast<uint32_t>(h * kBN),
                          a_base + soff + h * (16384u >> 4) + kk * a_step,
                          b_base + soff + kk * b_step, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        };
        if (kOrderable && g.ordered) {
          // Ordered drain (the epilogue releases half 0's TMEM columns, then half 1's): the
          // tile starts on half 0 alone, and half 1's MMAs trail by the stages filled before
          // half 1 was released (at most the ring's depth), so the tensor pipe works through
          // the second half of the previous tile's epilogue. Each stage is released once both
          // halves have used it. Every accumulator element still sums its K slices in order.
          bool h1_free = false;
          int lag = 0;            // first K block whose half-1 MMAs are not issued yet
          int lag_stage = stage;  // its ring stage
          for (int kb = 0; kb < k_blocks; ++kb) {
            if (!mbar_wait(full_bar(stage), phase, g.status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_half(stage, 0, kb);
            if (!h1_free) {
              if (kb + 1 - lag == kPairStages || kb + 1 == k_blocks) {
                // every stage waits for half 1, or the tile ends: wait for the release
                if (!mbar_wait_cluster(tempty_bar(1), acc_phase ^ 1u, g.status, abort_flag)) {
                  ok = false;
                  break;
                }
                h1_free = true;
              } else {
                h1_free = mbar_test_cluster(tempty_bar(1), acc_phase ^ 1u) != 0;
              }
              if (h1_free) tc_fence_after_sync();
            }
            if (h1_free) {
              for (; lag <= kb; ++lag) {
                issue_half(lag_stage, 1, lag);
                mma_commit_pair(empty_bar(lag_stage), 0x3);
                ++consumed;
                if (++lag_stage == kPairStages) lag_stage = 0;
              }
            }
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        } else {
          for (int kb = 0; kb < k_blocks; ++kb) {
            if (!mbar_wait(full_bar(stage), phase, g.status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint64_t soff = static_cast<uint64_t>(stage * kPairStageBytes) >> 4;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
              if constexpr (kTF32x3) {
                // corrections lo.hi + hi.lo into their own accumulator, then hi.hi
                const uint64_t a_hi = a_base + soff + kk * a_step;
                const uint64_t b_hi = b_base + soff + kk * b_step;
                const uint64_t a_lo = a_hi + (kPairABytes >> 4);
                const uint64_t b_lo = b_hi + (G::kBBytes >> 4);
                const uint32_t d_corr = d_tmem + static_cast<uint32_t>(kBN);
                mma_tf32_pair(d_corr, a_lo, b_hi, idesc, accum);
                mma_tf32_pair(d_corr, a_hi, b_lo, idesc, 1u);
                mma_tf32_pair(d_tmem, a_hi, b_hi, idesc, accum);
              } else {
#pragma unroll
                for (int h = 0; h < G::kHalves; ++h)
                  mma_bf16_pair(d_tmem + static_cast<uint32_t>(h * kBN),
                                a_base + soff + h * (16384u >> 4) + kk * a_step,
                                b_base + soff + kk * b_step, idesc, accum);
              }
            }
            mma_commit_pair(empty_bar(stage), 0x3);
            ++consumed;
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        // (g.withhold: the failure-path test leaves the first pair's first tile unsignalled so
        // that both CTAs' epilogue waits run out.)
        if (!(g.withhold && cluster_id == 0 && consumed == k_blocks))
          mma_commit_pair(tfull_bar(acc), 0x3);
        if (++acc == G::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      *consumed_fills = consumed;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    // Epilogue warp e = warp - 2 drains lane quarter warp % 4 (the quarter a warp may access)
    // of 128-row half (e / 4) % kHalves, column part e / (4 kHalves) of kSplit.
    const int quarter = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int half = grp % G::kHalves;
    const int part = grp / G::kHalves;
    const int row = quarter * 32 + lane;
    uint4* stage = reinterpret_cast<uint4*>(smem + kPairRingBytes + 1024 +
                                            static_cast<uint32_t>(warp - 2) * kEpiStageBytes);
    // the part-0 warp of this row block lends the exchange slots (epilogues that combine
    // per-row partials across the two parts do not use store staging)
    const int e_part0 = 4 * half + ((quarter - 2) & 3);
    float4* xchg = reinterpret_cast<float4*>(smem + kPairRingBytes + 1024 +
                                             static_cast<uint32_t>(e_part0) * kEpiStageBytes);
    // ordered drain: warp 2 + 4 p + (q - 2) % 4 takes column half p of lane quarter q in both
    // row halves; the part-0 warp lends its staging as 2 halves x 2 slots of 32 float4 (2 KB)
    float4* xchg_ordered = reinterpret_cast<float4*>(
        smem + kPairRingBytes + 1024 + static_cast<uint32_t>((quarter - 2) & 3) * kEpiStageBytes);
    static_assert(kEpiStageBytes >= 2 * 2 * 32 * sizeof(float4), "ordered-drain exchange slots");
    int acc = 0;
    uint32_t acc_phase = 0;
    typename Epi0::State st0;
    typename Epi1::State st1;
    Epi0::init(e0, st0);
    Epi1::init(e1, st1);
    int qslot = 0;
    uint32_t qphase = 0;
    int iter = 0;
    while (true) {
      if (!mbar_wait_cluster(tq_full(qslot), qphase, g.status, abort_flag)) break;
      const int t = tile_q[qslot];
      __syncwarp();
      if (lane == 0) tq_release(qslot);
      if (++qslot == kTileQueue) {
        qslot = 0;
        qphase ^= 1u;
      }
      if (t < 0) break;
      const TileInfo pt = map_tile(g, t);
      // Ordered drain: the 8 warps take column half `grp` of both 128-row halves, half 0
      // first, and release each half's TMEM columns as soon as it is drained (tempty_bar(h)),
      // so that the next tile's half-0 MMAs overlap the drain of half 1. Otherwise each warp
      // drains its own half and columns once and releases the accumulator (tempty_bar(acc)).
      const bool ordered = kOrderable && g.ordered;  // uniform
      const int n_pass = ordered ? 2 : 1;
      const int mb_first =
          (pt.mb * 2 + static_cast<int>(rank)) * G::kHalves + (ordered ? 0 : half);
      EpiRows rows0, rows1;  // the rows' inputs, loaded while the MMAs still run
      if (pt.prob == 0)
        Epi0::fetch(e0, mb_first, row, rows0);
      else
        Epi1::fetch(e1, mb_first, row, rows0);
      rows1 = rows0;
      if (ordered) {
        if (pt.prob == 0)
          Epi0::fetch(e0, mb_first + 1, row, rows1);
        else
          Epi1::fetch(e1, mb_first + 1, row, rows1);
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, g.status, abort_flag)) break;
      tc_fence_after_sync();
      __syncwarp();
#pragma unroll 1
      for (int pass = 0; pass < n_pass; ++pass) {
        const int h = ordered ? pass : half;
        const int col_part = ordered ? grp : part;
        const int mb128 = mb_first + pass;
        EpiCtx ctx;
        ctx.row = row;
        ctx.taddr = tmem_base + static_cast<uint32_t>((acc * G::kHalves + h) * kBN) +
                    (static_cast<uint32_t>(quarter * 32) << 16);
        ctx.stage = stage;
        ctx.split = ordered ? 2 : kSplit;
        ctx.c_begin = col_part * (kBN / 32 / ctx.split);
        ctx.c_end = ctx.c_begin + kBN / 32 / ctx.split;
        ctx.part = col_part;
        ctx.iter = iter;
        ctx.two_acc = kTF32x3 ? 1 : 0;
        ctx.taddr_corr = ctx.taddr + static_cast<uint32_t>(kBN);  // 3xTF32: the corrections
        ctx.xbar = x_bar(quarter + 4 * h);
        ctx.xchg = ordered ? xchg_ordered + 64 * h : xchg;
        ctx.status = g.status;
        ctx.abort = abort_flag;
        ctx.rows = pass == 0 ? rows0 : rows1;
        if (pt.prob == 0)
          Epi0::tile(e0, st0, mb128, pt.nb, ctx);
        else
          Epi1::tile(e1, st1, mb128, pt.nb, ctx);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_cta(mapa_shared(tempty_bar(ordered ? h : acc), 0));
      }
      ++iter;
      if (++acc == G::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out of time somewhere in this CTA. Let in-flight work land before the pair's
    // shared memory and TMEM go away: the leader drains its MMAs and waits for the fills it
    // armed (they include the peer's bytes); the peer gives its own copies time to complete.
    if (warp == 1 && lane == 0 && leader) {
      mma_commit_pair(drain_bar(), 0x1);
      mbar_wait_bounded(drain_bar(), 0u);
    }
    if (warp == 0 && lane == 0) {
      if (leader) {
        const int issued = *issued_fills;
        for (int f = *consumed_fills; f < issued; ++f)
          mbar_wait_bounded(full_bar(f % kPairStages),
                            static_cast<uint32_t>((f / kPairStages) & 1));
      } else {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
    __syncthreads();
  }
  cluster_sync_all();  // no CTA leaves while its peer may still read its smem or signal it
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------- host helpers

// How many CTA pairs of `kern` can be resident at once on the current device (queried once
// per device and kernel). Depends on how the chip's SMs are grouped, not only on their count.
template <int kRows, int kSplit, bool kTF32x3 = false, class K>
int pair_resident_clusters(K kern, int sms) {
  using G = PairGeom<kRows, kSplit, kTF32x3>;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return sms / 2;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(G::kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear the query's error; fall back to one pair per two SMs
    n = sms / 2;
  }
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

// Launch one or two problems on CTA pairs: a persistent grid of as many pairs as can be
// resident at once (at most one per tile). The problems' m_tiles count PairGeom<kRows>::
// kTileRows-row tiles, and K-major A operands are boxed {64 x kRows}.
template <int kRows, int kSplit, class Epi0, class Epi1, bool kTF32x3 = false>
cudaError_t launch_pair(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
                        const CUtensorMap& b1, GemmGrid g, const typename Epi0::Args& e0,
                        const typename Epi1::Args& e1, int sms, cudaStream_t stream) {
  using G = PairGeom<kRows, kSplit, kTF32x3>;
  auto kern = k_umma_gemm_pair<kRows, kSplit, Epi0, Epi1, kTF32x3>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int max_clusters = pair_resident_clusters<kRows, kSplit, kTF32x3>(kern, sms);
  finish_grid(g);
  if (g.tile_counter) {
    e = cudaMemsetAsync(g.tile_counter, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
  }
  g.withhold = take_withhold_request() ? 1 : 0;
  const int clusters = g.num_tiles < max_clusters ? g.num_tiles : max_clusters;
  kern<<<2 * clusters, G::kThreads, G::kSmemBytes, stream>>>(a0, b0, a1, b1, g, e0, e1);
  return cudaGetLastError();
}

// Launch on a pair core (kCorePair: 128-row CTA tiles, kCoreWide: 256-row CTA tiles); the
// problems must have been made with core_tile_rows(core). kSplitWide: epilogue warps per row
// block on the wide core (2 for roles whose epilogues fit the smaller register budget of 576
// threads, when `role` is in the tune_split_epilogue() mask). Otherwise wide tiles of a role in
// the tune_ordered_drain() mask drain their two row halves one after the other.
template <class Epi0, class Epi1, int kSplitWide = 1>
cudaError_t launch_pair_core(Core core, const CUtensorMap& a0, const CUtensorMap& b0,
                             const CUtensorMap& a1, const CUtensorMap& b1, GemmGrid g,
                             const typename Epi0::Args& e0, const typename Epi1::Args& e1, int sms,
                             cudaStream_t stream, int role = 0) {
  g.ordered = 0;
  if (core == kCoreWide) {
    if (kSplitWide == 2 && (tune_split_epilogue() & role) != 0)
      return launch_pair<256, kSplitWide, Epi0, Epi1>(a0, b0, a1, b1, g, e0, e1, sms, stream);
    g.ordered = (tune_ordered_drain() & role) != 0 ? 1 : 0;
    return launch_pair<256, 1, Epi0, Epi1>(a0, b0, a1, b1, g, e0, e1, sms, stream);
  }
  return launch_pair<128, 1, Epi0, Epi1>(a0, b0, a1, b1, g, e0, e1, sms, stream);
}

// fp32 (3xTF32) problem on CTA pairs with 128-row CTA tiles (256 x 256 pair tiles): every
// operand K-major, a_hi / b_hi the TF32 hi copies and a_lo / b_lo the lo copies; A maps boxed
// {32 x 128}, B maps {32 x 128} (one CTA's N half); the problem made with 256-row tiles and
// 32-deep K blocks.
template <class Epi>
cudaError_t launch_pair_tf32(const CUtensorMap& a_hi, const CUtensorMap& b_hi,
                             const CUtensorMap& a_lo, const CUtensorMap& b_lo, GemmGrid g,
                             const typename Epi::Args& e, int sms, cudaStream_t stream) {
  g.ordered = 0;
  return launch_pair<128, 1, Epi, NoEpi, true>(a_hi, b_hi, a_lo, b_lo, g, e, NoEpi::Args{}, sms,
                                               stream);
}

}  // namespace flce
