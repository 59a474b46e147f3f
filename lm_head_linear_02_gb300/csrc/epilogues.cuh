// epilogues.cuh - what each FLCE kernel does with a finished 128 x 256 block of fp32
// accumulators (one tile on the single-SM core; one CTA's share, or one half of it, on pairs).
//
// Every epilogue thread owns one accumulator row (one TMEM lane) and walks its 256 columns in
// eight 32-column chunks (tcgen05.ld 32x32b.x32), so the per-row reductions of the softmax are
// plain in-thread loops with no cross-thread traffic.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "gemm.cuh"

namespace flce {

constexpr float kLog2e = 1.4426950408889634f;

// Columns [32c, 32c + 32) of this warp's rows of the finished tile: one accumulator, or the
// fp32 sum of the large and the correction accumulator (3xTF32 path).
__device__ __forceinline__ void load_chunk(const EpiCtx& ctx, int c, float (&v)[32]) {
  __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp issues it together
  uint32_t r[32];
  tmem_ld32(ctx.taddr + static_cast<uint32_t>(c * 32), r);
  if (ctx.two_acc) {  // uniform
    uint32_t q[32];
    tmem_ld32(ctx.taddr_corr + static_cast<uint32_t>(c * 32), q);
    tmem_ld_wait(r);
    tmem_ld_wait(q);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) + __uint_as_float(q[j]);
    return;
  }
  tmem_ld_wait(r);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Store 32 consecutive fp32 values as bf16 (64 bytes, 16-byte aligned destination), or only
// the first `n` (a multiple of 8) of them.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&v)[32], int n) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q * 8 < n) {
      uint4 w;
      w.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
      w.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
      w.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
      w.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
      d[q] = w;
    }
  }
}

// Store up to 32 fp32 values (n a multiple of 4, destination 16-byte aligned).
__device__ __forceinline__ void store_f32x32(float* dst, const float (&v)[32], int n) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (q * 4 < n) d[q] = make_float4(v[q * 4 + 0], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
}

// Exchange a warp's block of 32 rows x 64 bytes, held one row per lane (in[k] = bytes
// [16k, 16k + 16) of lane r's row), so that lane 4a + b ends with out[q] = bytes [16b, 16b + 16)
// of row 8q + a: afterwards each warp-wide 16-byte access covers 8 rows x 64 contiguous bytes
// instead of 32 scattered 16-byte pieces. The block passes through the warp's 2 KB of shared
// memory with its 16-byte units XOR-swizzled by row, so that the writes and the transposed
// reads are both free of bank conflicts. Every lane of the warp must call this.
__device__ __forceinline__ void transpose_rows64(uint4* stage, const uint4 (&in)[4],
                                                 uint4 (&out)[4], int lane) {
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) stage[lane * 4 + (k ^ sw)] = in[k];
  __syncwarp();
  const int a = lane >> 2, b = lane & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = 8 * q + a;
    out[q] = stage[r * 4 + (b ^ ((r >> 1) & 3))];
  }
  __syncwarp();  // the next block may overwrite the staging area
}

// Store 32 rows x 32 bf16 columns held one row per lane (value j of lane r at row row0 + r,
// column j of `base`) through transpose_rows64. Rows at or beyond `nrows` are not stored.
__device__ __forceinline__ void store_rows_bf16x32(uint4* stage, const float (&v)[32], int lane,
                                                   __nv_bfloat16* base, size_t ld, int row0,
                                                   int nrows) {
  uint4 in[4], out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    in[k] = make_uint4(pack_bf16x2(v[8 * k + 0], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                       pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
  transpose_rows64(stage, in, out, lane);
  const int a = lane >> 2, b = lane & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = row0 + 8 * q + a;
    if (r < nrows) *reinterpret_cast<uint4*>(base + static_cast<size_t>(r) * ld + b * 8) = out[q];
  }
}

// TF32 split of an fp32 value: hi keeps the top 10 mantissa bits (rounded to nearest), and
// lo = x - hi is exact in fp32. hi + lo == x.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  uint32_t h;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
  hi = __uint_as_float(h);
  lo = x - hi;
}

// Maximum of 32 values in 16 three-input max instructions (exact: any order gives the same).
__device__ __forceinline__ float max32(const float (&v)[32]) {
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  t[10] = fmaxf(v[30], v[31]);
  return max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]),
              max3(max3(t[6], t[7], t[8]), t[9], t[10]));
}

// ------------------------------------------------------------------------------- forward
// "[example] fused_linear_cross_entropy kernel" (Helion PR #1268), forward: a tiled matmul
// feeding an online softmax that yields the log-sum-exp and the target logit of each row.
// Each (vocab tile, token) pair leaves a partial (max m, sum of exp(z - m)) that the combine
// kernel merges in a fixed order; the one tile holding target[t] also writes z[t, target[t]]
// and sx[t], its sum of exp(z - m) without the target column, from which the combine forms
// the per-token loss without cancellation when the target dominates its row. Vocab columns
// >= V are masked to -inf.
// A tile's partial is formed from its two 128-column halves (chunks 0-3 and 4-7), each folded
// chunk by chunk, then merged: half 1 into half 0. One warp does both halves, or two warps one
// each (split 2, half 1 passed to half 0's warp through the exchange slots); the arithmetic,
// and so every bit of the result, is the same either way.
struct FwdEpi {
  struct Args {
    const int64_t* target;
    float* part_m;  // [n_tiles][T], n_tiles = ceil(V_total / 256)
    float* part_s;  // [n_tiles][T]
    float* zy;      // [T]
    float* sx;      // [T]: the target tile's sum without the target column
    int T, V;       // V: vocab columns of this launch
    int col0;       // vocab column of the launch's first column (a multiple of 256)
  };
  struct State {};
  static __device__ __forceinline__ void init(const Args&, State&) {}
  static __device__ __forceinline__ void fetch(const Args& a, int mb, int row, EpiRows& r) {
    const int t = mb * kBM + row;
    r.y = t < a.T ? static_cast<long long>(a.target[t]) : -1ll;
  }

  // Fold chunks [c_begin, c_end) of the tile into (m, s); picks up the target logit. With
  // kExclude the target column's term is left out of s (the row's other columns are summed in
  // exactly the same order, so a row whose target lies elsewhere gets the same s either way).
  template <bool kExclude>
  static __device__ __forceinline__ void fold(const Args& a, const EpiCtx& ctx, int n0, int rel,
                                              int c_begin, int c_end, float& m, float& s,
                                              float& zy) {
    m = -INFINITY;
    s = 0.f;
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int c0 = n0 + c * 32;
      if (c0 >= a.V) break;  // uniform across the warp
      float v[32];
      load_chunk(ctx, c, v);
      if (c0 + 32 > a.V) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j >= a.V) v[j] = -INFINITY;
      }
      const int q = rel - c * 32;
      if (!kExclude && q >= 0 && q < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == q) zy = v[j];
      }
      const float mn = fmaxf(m, max32(v));
      const float mnl = mn * kLog2e;
      // four running sums (terms j, j+1, j+2, j+3 of each group of four), kept as two lane pairs
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float e0, e1, e2, e3;
        fma2(e0, e1, v[j + 0], v[j + 1], kLog2e, -mnl);
        fma2(e2, e3, v[j + 2], v[j + 3], kLog2e, -mnl);
        e0 = ex2(e0);
        e1 = ex2(e1);
        e2 = ex2(e2);
        e3 = ex2(e3);
        if (kExclude) {
          e0 = j + 0 == q ? 0.f : e0;
          e1 = j + 1 == q ? 0.f : e1;
          e2 = j + 2 == q ? 0.f : e2;
          e3 = j + 3 == q ? 0.f : e3;
        }
        add2(s0, s1, e0, e1);
        add2(s2, s3, e2, e3);
      }
      s = s * ex2((m - mn) * kLog2e) + ((s0 + s1) + (s2 + s3));
      m = mn;
    }
  }

  // Partial (m, s, sx) of chunks [c_begin, c_end): sx = s unless some row of the warp has its
  // target there, when the chunks are folded once more without the target column (a few
  // percent of tiles: the rows of a warp target 32 of the V / 256 tiles at most).
  static __device__ __forceinline__ void half_partial(const Args& a, const EpiCtx& ctx, int n0,
                                                      int rel, int c_begin, int c_end, float& m,
                                                      float& s, float& sx, float& zy) {
    fold<false>(a, ctx, n0, rel, c_begin, c_end, m, s, zy);
    sx = s;
    if (__any_sync(0xffffffffu, rel >= c_begin * 32 && rel < c_end * 32)) {
      float mx, unused = 0.f;
      fold<true>(a, ctx, n0, rel, c_begin, c_end, mx, sx, unused);
    }
  }

  // Merge half 1's partial into half 0's (half 1 may be empty: -inf, 0, 0).
  static __device__ __forceinline__ void merge(float& m0, float& s0, float& sx0, float m1,
                                               float s1, float sx1) {
    const float mn = fmaxf(m0, m1);
    const float f0 = ex2((m0 - mn) * kLog2e), f1 = ex2((m1 - mn) * kLog2e);
    s0 = s0 * f0 + s1 * f1;
    sx0 = sx0 * f0 + sx1 * f1;
    m0 = mn;
  }

  static __device__ __forceinline__ void tile(const Args& a, State&, int mb, int nb,
                                              const EpiCtx& ctx) {
    const int t = mb * kBM + ctx.row;
    const bool valid = t < a.T;
    const int n0 = nb * kBN;  // launch-relative column of the tile
    const long long y = valid ? ctx.rows.y - a.col0 : -1ll;
    const int rel = (y >= n0 && y < n0 + kBN) ? static_cast<int>(y - n0) : -1;
    constexpr int kHalfChunks = kBN / 64;
    float zy = 0.f;
    float m, s, sx;
    if (ctx.split == 1) {
      float m1, s1, sx1;
      half_partial(a, ctx, n0, rel, 0, kHalfChunks, m, s, sx, zy);
      half_partial(a, ctx, n0, rel, kHalfChunks, 2 * kHalfChunks, m1, s1, sx1, zy);
      merge(m, s, sx, m1, s1, sx1);
    } else {
      half_partial(a, ctx, n0, rel, ctx.c_begin, ctx.c_end, m, s, sx, zy);
      float4* slot = ctx.xchg + 32 * (ctx.iter & 1);
      const int lane = ctx.row & 31;
      if (ctx.part == 1) {
        slot[lane] = make_float4(m, s, sx, 0.f);
        mbar_arrive(ctx.xbar);
      } else {
        if (!mbar_wait(ctx.xbar, static_cast<uint32_t>(ctx.iter & 1), ctx.status, ctx.abort))
          return;  // the partner left on the abort path: outputs are undefined anyway
        const float4 o = slot[lane];
        merge(m, s, sx, o.x, o.y, o.z);
      }
    }
    if (valid && ctx.part == 0) {
      const size_t o = static_cast<size_t>(a.col0 / kBN + nb) * a.T + t;
      a.part_m[o] = m;
      a.part_s[o] = s;
      if (rel >= 0) a.sx[t] = sx;
    }
    if (valid && rel >= ctx.c_begin * 32 && rel < ctx.c_end * 32) a.zy[t] = zy;
  }
};

// ------------------------------------------------------------------------------- chunk logits
// Single-call forward + backward over a chunk of tokens (the logits are computed once, not
// recomputed): like FwdEpi, each (128-column vocab half-tile, token) pair leaves its (max m, sum
// of exp(z - m)) partial and the half-tile holding target[t] writes z[t, target[t]] and its sum
// without the target column; in addition the
// half-tile's logits are kept, shifted by their maximum, as bf16 in a chunk buffer
// zbuf[t][v] = z[t, v] - m. The shift puts the largest logits of each half-tile near 0, where
// bf16 is most precise, so exp(zbuf + m - lse) recovers the dominant softmax terms accurately.
// Two passes over each half's TMEM columns: its maximum first, then the shifted store and the
// exp-sum. One warp does both halves, or two warps one each (split 2); every partial belongs
// to one half, so nothing is exchanged and the results do not depend on the split.
struct LogitsEpi {
  struct Args {
    const int64_t* target;  // chunk rows
    float* part_m;          // [2 n_tiles][T]: one partial per 128-column half-tile
    float* part_s;          // [2 n_tiles][T]
    float* zy;              // [T]
    float* sx;              // [T]: the target half-tile's sum without the target column
    __nv_bfloat16* zbuf;    // [T][ldz]
    int ldz;
    int T, V;
  };
  struct State {};
  static __device__ __forceinline__ void init(const Args&, State&) {}
  static __device__ __forceinline__ void fetch(const Args& a, int mb, int row, EpiRows& r) {
    const int t = mb * kBM + row;
    r.y = t < a.T ? static_cast<long long>(a.target[t]) : -1ll;
  }

  static __device__ __forceinline__ void half(const Args& a, const EpiCtx& ctx, int t, bool valid,
                                              int nb, int rel, int h) {
    constexpr int kHalfChunks = kBN / 64;
    const int n0 = nb * kBN;
    float m = -INFINITY, zy = 0.f;
#pragma unroll 1
    for (int c = h * kHalfChunks; c < (h + 1) * kHalfChunks; ++c) {
      const int c0 = n0 + c * 32;
      if (c0 >= a.V) break;  // uniform across the warp
      float v[32];
      load_chunk(ctx, c, v);
      const int q = rel - c * 32;
      if (c0 + 32 <= a.V) {  // uniform
        m = fmaxf(m, max32(v));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < a.V) m = fmaxf(m, v[j]);
      }
      if (q >= 0 && q < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == q) zy = v[j];
      }
    }
    const float ml = m * kLog2e;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
    for (int c = h * kHalfChunks; c < (h + 1) * kHalfChunks; ++c) {
      const int c0 = n0 + c * 32;
      if (c0 >= a.V) break;
      float v[32];
      load_chunk(ctx, c, v);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float e0, e1;
        fma2(e0, e1, v[j], v[j + 1], kLog2e, -ml);
        e0 = ex2(e0);
        e1 = ex2(e1);
        add2(s0, s1, (c0 + j < a.V) ? e0 : 0.f, (c0 + j + 1 < a.V) ? e1 : 0.f);
        fma2(v[j], v[j + 1], v[j], v[j + 1], 1.0f, -m);  // v - m, rounded once
      }
      store_rows_bf16x32(ctx.stage, v, ctx.row & 31, a.zbuf + c0, a.ldz, t - (ctx.row & 31),
                         a.T);
    }
    const bool mine = rel >= h * 128 && rel < (h + 1) * 128;
    float x0 = s0, x1 = s1;  // the sum without the target column (rows whose target is here)
    if (__any_sync(0xffffffffu, mine)) {
      x0 = 0.f;
      x1 = 0.f;
#pragma unroll 1
      for (int c = h * kHalfChunks; c < (h + 1) * kHalfChunks; ++c) {
        const int c0 = n0 + c * 32;
        if (c0 >= a.V) break;
        float v[32];
        load_chunk(ctx, c, v);
        const int q = rel - c * 32;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float e0 = ex2(fmaf(v[j], kLog2e, -ml));
          const float e1 = ex2(fmaf(v[j + 1], kLog2e, -ml));
          x0 += (c0 + j < a.V && j != q) ? e0 : 0.f;
          x1 += (c0 + j + 1 < a.V && j + 1 != q) ? e1 : 0.f;
        }
      }
    }
    if (valid) {
      const size_t o = static_cast<size_t>(2 * nb + h) * a.T + t;
      a.part_m[o] = m;
      a.part_s[o] = s0 + s1;
      if (mine) {
        a.zy[t] = zy;
        a.sx[t] = x0 + x1;
      }
    }
  }

  static __device__ __forceinline__ void tile(const Args& a, State&, int mb, int nb,
                                              const EpiCtx& ctx) {
    const int t = mb * kBM + ctx.row;
    const bool valid = t < a.T;
    const int n0 = nb * kBN;
    const long long y = valid ? ctx.rows.y : -1ll;
    const int rel = (y >= n0 && y < n0 + kBN) ? static_cast<int>(y - n0) : -1;
    if (ctx.split == 1) {
      half(a, ctx, t, valid, nb, rel, 0);
      half(a, ctx, t, valid, nb, rel, 1);
    } else {
      half(a, ctx, t, valid, nb, rel, ctx.part);
    }
  }
};

// ------------------------------------------------------------------------------- backward dz
// "[example] fused_linear_cross_entropy kernel" (Helion PR #1268), backward: the logits are
// recomputed and turned into dz = (softmax - onehot(target)) * g in registers; here the
// unscaled factor (softmax - onehot), whose entries lie in [-1, 1], is written to a bounded
// vocab slab (T x Vc) that feeds the two gradient contractions, and g is applied in fp32 in
// their epilogues. Keeping g out of the bf16 slab keeps the dominant -1 entries exact for the
// 'sum' and 'mean' reductions. With per-token upstream gradients ('none' reduction) each row is
// multiplied by its own g[t] here instead (row_scale), since grad_W sums over the rows.
// Columns outside the slab are stored as 0; rows >= T are not stored.
template <bool kTF32>
struct DzEpi {
  struct Args {
    const int64_t* target;
    const float* lse;
    const float* row_scale;  // per-token upstream gradient [T], or null (factor 1)
    void* dz;      // bf16 [T][ldz] or fp32 hi [T][ldz]
    float* dz_lo;  // fp32 lo [T][ldz]          (tf32)
    float* dzt_hi; // fp32 [slab_w][ldt]        (tf32)
    float* dzt_lo; // fp32 [slab_w][ldt]        (tf32)
    int ldz, ldt;
    int T, slab0, slab_w;
  };
  struct State {};
  static __device__ __forceinline__ void init(const Args&, State&) {}
  static __device__ __forceinline__ void fetch(const Args& a, int mb, int row, EpiRows& r) {
    const int t = mb * kBM + row;
    const bool valid = t < a.T;
    r.y = valid ? static_cast<long long>(__ldg(a.target + t)) : -1ll;
    r.lse = valid ? __ldg(a.lse + t) : 0.f;
    r.scale = (valid && a.row_scale) ? __ldg(a.row_scale + t) : 1.0f;
  }

  static __device__ __forceinline__ void tile(const Args& a, State&, int mb, int nb,
                                              const EpiCtx& ctx) {
    const int row = ctx.row;
    uint4* stage = ctx.stage;
    const int t = mb * kBM + row;
    const bool valid = t < a.T;
    const float lsel = ctx.rows.lse * kLog2e;
    const long long y = ctx.rows.y;
    const float rs = ctx.rows.scale;
    const int n0 = nb * kBN;  // slab-relative column of the tile
    const long long rel = y - a.slab0 - n0;
    const bool unit_scale = a.row_scale == nullptr;  // uniform: sum / mean reductions
#pragma unroll 1
    for (int c = ctx.c_begin; c < ctx.c_end; ++c) {
      const int c0 = n0 + c * 32;
      if (c0 >= a.slab_w) break;  // uniform
      float v[32];
      load_chunk(ctx, c, v);
      if (unit_scale && c0 + 32 <= a.slab_w) {
        // The common case: every column inside the slab and row factor 1, so only the one
        // target column of a row (if it lies in this chunk) differs from exp(z - lse).
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          fma2(v[j], v[j + 1], v[j], v[j + 1], kLog2e, -lsel);
          v[j] = ex2(v[j]);
          v[j + 1] = ex2(v[j + 1]);
        }
        const long long q = rel - c * 32;
        if (q >= 0 && q < 32) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == q) v[j] -= 1.0f;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float d = ex2(fmaf(v[j], kLog2e, -lsel));
          if (rel == c * 32 + j) d -= 1.0f;
          if (c0 + j >= a.slab_w) d = 0.f;
          v[j] = d * rs;
        }
      }
      if constexpr (!kTF32) {
        store_rows_bf16x32(stage, v, row & 31, reinterpret_cast<__nv_bfloat16*>(a.dz) + c0,
                           static_cast<size_t>(a.ldz), t - (row & 31), a.T);
      } else {
        if (!valid) continue;
        float hi[32], lo[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) split_tf32(v[j], hi[j], lo[j]);
        store_f32x32(reinterpret_cast<float*>(a.dz) + static_cast<size_t>(t) * a.ldz + c0, hi, 32);
        store_f32x32(a.dz_lo + static_cast<size_t>(t) * a.ldz + c0, lo, 32);
        // Transposed copies: column c0 + j of this row goes to row c0 + j, column t. A warp's
        // 32 lanes hold 32 consecutive t, so each of these stores is one coalesced 128 B line.
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (c0 + j < a.slab_w) {
            a.dzt_hi[static_cast<size_t>(c0 + j) * a.ldt + t] = hi[j];
            a.dzt_lo[static_cast<size_t>(c0 + j) * a.ldt + t] = lo[j];
          }
        }
      }
    }
  }
};

// ------------------------------------------------------------------------------- grad_weight
// grad_weight[slab rows, :] = dz_slab^T . x : the contraction runs over all T tokens, so each
// output tile is complete when it leaves TMEM and is written exactly once.
// The accumulator holds (softmax - onehot)^T . x; the gradient scale g = grad_loss (sum) or
// grad_loss / T (mean) is applied here in fp32 (grad_loss null: g = scale, the 'none' case whose
// per-token factors are already in the dz rows).
template <bool kF32Out>
struct GradWEpi {
  struct Args {
    void* grad_w;  // [V][H]
    const float* grad_loss;
    float scale;
    int H, slab0, slab_w;
  };
  struct State {
    float g;
  };
  static __device__ __forceinline__ void init(const Args& a, State& st) {
    st.g = a.grad_loss ? __ldg(a.grad_loss) * a.scale : a.scale;
  }
  static __device__ __forceinline__ void fetch(const Args&, int, int, EpiRows&) {}

  static __device__ __forceinline__ void tile(const Args& a, State& st, int mb, int nb,
                                              const EpiCtx& ctx) {
    const int row = ctx.row;
    uint4* stage = ctx.stage;
    const int r = mb * kBM + row;  // slab-relative vocab row
    const bool valid = r < a.slab_w;
    const size_t vrow = static_cast<size_t>(a.slab0) + r;
    const int lane = row & 31;
#pragma unroll 1
    for (int c = ctx.c_begin; c < ctx.c_end; ++c) {
      const int h0 = nb * kBN + c * 32;
      if (h0 >= a.H) break;
      float v[32];
      load_chunk(ctx, c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= st.g;
      if constexpr (kF32Out) {
        if (valid) store_f32x32(reinterpret_cast<float*>(a.grad_w) + vrow * a.H + h0, v,
                                min(32, a.H - h0));
      } else {
        // 8 bf16 columns per 16-byte unit; H is a multiple of 8, so units are whole or absent
        uint4 in[4], out[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          in[k] = make_uint4(pack_bf16x2(v[8 * k + 0], v[8 * k + 1]),
                             pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                             pack_bf16x2(v[8 * k + 4], v[8 * k + 5]),
                             pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
        transpose_rows64(stage, in, out, lane);
        const int qa = lane >> 2, qb = lane & 3;
        const int r0 = r - lane;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int rr = r0 + 8 * q + qa;
          const int col = h0 + qb * 8;
          if (rr < a.slab_w && col < a.H)
            *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.grad_w) +
                                      (static_cast<size_t>(a.slab0) + rr) * a.H + col) = out[q];
        }
      }
    }
  }
};

// ------------------------------------------------------------------------------- grad_x
// grad_x = sum over vocab slabs of dz_slab . W_slab: a split-K over the vocabulary whose parts
// are added in slab order into an fp32 accumulator (deterministic; no atomics).
//   mode 0: only slab   -> out = D
//   mode 1: first slab  -> acc = D
//   mode 2: middle slab -> acc += D
//   mode 3: last slab   -> out = acc + D
//   mode 4: out += D, read and rounded back in the output type (bf16 outputs only): the
//           single call's grad_weight summed over token chunks in its own output buffer
// For fp32 outputs `acc` and `out` are the same buffer.
// As for grad_W, the slab product is scaled by g in fp32 before it is accumulated.
template <bool kF32Out>
struct GradXEpi {
  struct Args {
    float* acc;   // [T][H] fp32
    void* out;    // [T][H] dtype
    const float* grad_loss;
    float scale;
    int T, H, mode;
  };
  struct State {
    float g;
  };
  static __device__ __forceinline__ void init(const Args& a, State& st) {
    st.g = a.grad_loss ? __ldg(a.grad_loss) * a.scale : a.scale;
  }
  static __device__ __forceinline__ void fetch(const Args&, int, int, EpiRows&) {}

  static __device__ __forceinline__ void tile(const Args& a, State& st, int mb, int nb,
                                              const EpiCtx& ctx) {
    const int row = ctx.row;
    uint4* stage = ctx.stage;
    const int t = mb * kBM + row;
    const bool valid = t < a.T;
    if constexpr (!kF32Out) {
      // Each 32-column chunk in two 16-column halves of fp32 (64 bytes per row), transposed
      // through shared memory: lane 4a + b then owns columns [4b, 4b + 4) of rows 8q + a, and
      // every accumulator read, accumulator write and output store is coalesced.
      const int lane = row & 31;
      const int qa = lane >> 2, qb = lane & 3;
      const int t0 = t - lane;
#pragma unroll 1
      for (int c = ctx.c_begin; c < ctx.c_end; ++c) {
        const int h0 = nb * kBN + c * 32;
        if (h0 >= a.H) break;
        float v[32];
        load_chunk(ctx, c, v);
        // both 16-column halves through shared memory first, then every accumulator load of
        // the chunk in flight at once, then the adds and stores
        uint4 out[2][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint4 in[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            in[k] = make_uint4(__float_as_uint(v[16 * hh + 4 * k + 0] * st.g),
                               __float_as_uint(v[16 * hh + 4 * k + 1] * st.g),
                               __float_as_uint(v[16 * hh + 4 * k + 2] * st.g),
                               __float_as_uint(v[16 * hh + 4 * k + 3] * st.g));
          transpose_rows64(stage, in, out[hh], lane);
        }
        float4 p[2][4];
        if (a.mode == 2 || a.mode == 3) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int tr = t0 + 8 * q + qa;
              const int col = h0 + 16 * hh + 4 * qb;  // H is a multiple of 8: 4-column units
              p[hh][q] = (tr < a.T && col < a.H)
                             ? *reinterpret_cast<const float4*>(a.acc + static_cast<size_t>(tr) * a.H + col)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else if (a.mode == 4) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int tr = t0 + 8 * q + qa;
              const int col = h0 + 16 * hh + 4 * qb;
              uint2 u = make_uint2(0u, 0u);
              if (tr < a.T && col < a.H)
                u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.out) +
                                                    static_cast<size_t>(tr) * a.H + col);
              p[hh][q] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
            }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int tr = t0 + 8 * q + qa;
            const int col = h0 + 16 * hh + 4 * qb;
            if (tr >= a.T || col >= a.H) continue;
            const size_t o = static_cast<size_t>(tr) * a.H + col;
            float4 d = make_float4(__uint_as_float(out[hh][q].x), __uint_as_float(out[hh][q].y),
                                   __uint_as_float(out[hh][q].z), __uint_as_float(out[hh][q].w));
            if (a.mode >= 2) {
              d.x += p[hh][q].x;
              d.y += p[hh][q].y;
              d.z += p[hh][q].z;
              d.w += p[hh][q].w;
            }
            if (a.mode == 1 || a.mode == 2) {
              *reinterpret_cast<float4*>(a.acc + o) = d;
            } else {
              uint2 w;
              w.x = pack_bf16x2(d.x, d.y);
              w.y = pack_bf16x2(d.z, d.w);
              *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + o) = w;
            }
          }
      }
    } else {  // fp32 outputs (the TF32 path): plain per-row stores
#pragma unroll 1
      for (int c = ctx.c_begin; c < ctx.c_end; ++c) {
        const int h0 = nb * kBN + c * 32;
        if (h0 >= a.H) break;
        float v[32];
        load_chunk(ctx, c, v);
        if (!valid) continue;
        const int n = min(32, a.H - h0);
        const size_t o = static_cast<size_t>(t) * a.H + h0;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= st.g;
        if (a.mode >= 2) {
          const float4* s = reinterpret_cast<const float4*>(a.acc + o);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (q * 4 < n) {
              const float4 p = s[q];
              v[q * 4 + 0] += p.x;
              v[q * 4 + 1] += p.y;
              v[q * 4 + 2] += p.z;
              v[q * 4 + 3] += p.w;
            }
          }
        }
        store_f32x32((a.mode == 1 || a.mode == 2) ? a.acc + o : reinterpret_cast<float*>(a.out) + o,
                     v, n);
      }
    }
  }
};

}  // namespace flce
