// Pieces shared by the grouped GEMM kernels (per-token scales in gemm.cu,
// 128 x 128 block scales in gemm_block.cu): tile geometry, the tile table
// built on the device from the expert offsets, named-barrier helpers and the
// TMA descriptor cache.
//
// A tile is (expert, weight block, token chunk): 128 weight rows (the MMA's
// M side) against up to BNMAX of the expert's tokens (its N side). An
// expert's tokens are split into equal chunks, multiples of 16, and the tile
// index runs token chunk fastest so the chunks that read one weight block
// run side by side and share it through L2.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace gemm_common {

constexpr int BM = 128;   // weight rows per tile (MMA M)
constexpr int BK = 128;   // K bytes (= e4m3 elements) per K chunk
constexpr int W_BYTES = BM * BK;
constexpr int MAX_E = 1024;
constexpr uint64_t WAIT_NS = 2000000000ull;   // bound of every pipeline wait
constexpr uint64_t DRAIN_NS = 200000000ull;   // bound of the waits after a timeout

// Token boxes of 64/32/16 rows: a tile's tokens (rounded up to 16) are
// covered exactly by 64-row boxes plus at most one 32- and one 16-row box
// (64-row token boxes measured faster than 128-row ones).
constexpr int NXBOX = 3;
// Weights. When Kd is a multiple of 128 the weights of a pipeline stage move
// in one box: K is viewed as (128-byte chunk, chunk index) so that one box
// holds the stage's KC chunks, each landing as its own [rows][128 B] block.
// bf16 epilogue: [Kd/128][E*N][128], the tile's 128 rows per chunk. SiLU:
// [E][Kd/128][2][I][128], 64 gate rows then the matching 64 up rows per chunk
// (rows past I read as 0). Otherwise (the view would run into the next row)
// one box per chunk over [E*N][Kd] or [E][2][I][Kd], zero past Kd. Fewer
// copies per stage measured faster: one box per stage instead of two 64-row
// boxes per chunk took DeepSeek-V3 prefill w13 from 1.96 to 1.69 ms.
struct Maps {
  CUtensorMap w;           // weights (see above; SiLU: 5-D or 4-D, bf16: 3-D or 2-D)
  CUtensorMap x[NXBOX];    // tokens: box rows 64 >> i
  CUtensorMap xg;          // token-order rows [T, Kd], box one row high (gather4)
};

template <int BNMAX>
struct TileInfo {
  int e, nb, tok0, ntok;
  int nch;  // token chunks of the expert (1: the weight block is read by this tile only)
};

// tile -> (expert, weight block, token chunk)
template <int BNMAX, class S>
__device__ __forceinline__ TileInfo<BNMAX> decode_tile(const S& sm, int E, int NB, int tile) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo<BNMAX> t;
  t.e = lo;
  const int local = tile - sm.tile_start[lo];
  const int nch = (sm.tile_start[lo + 1] - sm.tile_start[lo]) / NB;
  t.nb = local / nch;
  t.nch = nch;
  const int tc = local - t.nb * nch;
  // equal chunks (multiples of 16 tokens) so the tiles that share a weight
  // block run at the same speed and meet it in L2
  const int cnt = sm.offs[lo + 1] - sm.offs[lo];
  const int csz = ((cnt + nch - 1) / nch + 15) & ~15;
  t.tok0 = sm.offs[lo] + tc * csz;
  t.ntok = min(csz, cnt - tc * csz);
  return t;
}

__device__ __forceinline__ void bar_sync_named(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also returns whether any participating thread passed a
// non-zero `pred`.
__device__ __forceinline__ int bar_red_or(int id, int count, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(count)
      : "memory");
  return r;
}


// Builds sm.offs[0..E], sm.tile_start[0..E] and sm.total_tiles (0 when the
// offsets are not monotone within [0, M], with MOE_DEV_BAD_OFFSETS raised)
// for NBG weight-block groups per expert and token chunks of at most BNMAX.
// Called by all THREADS threads; the caller synchronises before reading.
template <int BNMAX, int THREADS, class S>
__device__ __forceinline__ void build_tile_table(S& sm, const int32_t* offsets, int E, int M,
                                                 int NBG, int* err, int tid) {
  for (int i = tid; i <= E; i += THREADS) sm.offs[i] = __ldg(offsets + i);
  __syncthreads();
  const int per = (E + THREADS - 1) / THREADS;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  int bad = 0;
  for (int e = e0; e < e1; ++e) {
    const int lo = sm.offs[e], hi = sm.offs[e + 1];
    if (lo < 0 || hi < lo || hi > M) bad = 1;
    else local += (hi - lo + BNMAX - 1) / BNMAX;
  }
  // exclusive prefix of the per-thread tile counts: a shuffle scan in each
  // warp, then one over the warp totals
  static_assert(THREADS % 32 == 0 && THREADS <= 32 * 32, "block shape");
  constexpr int NW = THREADS / 32;
  const int lane = tid & 31, wid = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.thr_sum[wid] = incl;
  bad = __syncthreads_or(bad);
  if (wid == 0) {
    const int w = lane < NW ? sm.thr_sum[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += y;
    }
    __syncwarp();
    if (lane < NW) sm.thr_sum[lane] = wi - w;  // tiles before warp `lane`
    if (lane == NW - 1) {
      sm.total_tiles = bad ? 0 : wi * NBG;
      sm.tile_start[E] = wi * NBG;
      if (bad) flag_error(err, MOE_DEV_BAD_OFFSETS);
    }
  }
  __syncthreads();
  int run = sm.thr_sum[wid] + incl - local;
  for (int e = e0; e < e1; ++e) {
    sm.tile_start[e] = run * NBG;
    const int lo = sm.offs[e], hi = sm.offs[e + 1];
    if (!bad) run += (hi - lo + BNMAX - 1) / BNMAX;
  }
}

// Host: 2-D u8 tensor [rows, cols] (cols contiguous) with a box of 128 B x
// box_rows, 128-byte swizzle, zero fill outside the tensor. False when the
// driver cannot encode it.
bool make_tma_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows);

// Host: 2-D u8 tensor [rows, cols] with a box of 128 B x 1 row (128-byte
// swizzle, zero fill) for four-row gathers.
bool make_tma_map_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols);

// Host: weights [E, N, Kd] (Kd % 128 == 0), kc 128-byte K chunks of `rows`
// (<= 256) consecutive rows per box.
bool make_tma_map_weights_rows(CUtensorMap* m, const void* base, uint64_t E, uint64_t N,
                               uint64_t Kd, uint32_t rows, uint32_t kc = 1);

// Host: w13 [E, 2I, Kd] (Kd % 128 == 0) viewed per 128-byte K chunk, boxes of
// jrows (<= 256) gate rows followed by the matching jrows up rows, for kc
// consecutive chunks.
bool make_tma_map_weights_gateup(CUtensorMap* m, const void* base, uint64_t E, uint64_t N,
                                 uint64_t Kd, uint32_t jrows, uint32_t kc = 1);

// Host: w13 [E, 2I, Kd] (Kd % 128 == 0) viewed per 128-byte K chunk, boxes of
// 32 gate rows followed by the matching 32 up rows.
bool make_tma_map_weights_pairs32(CUtensorMap* m, const void* base, uint64_t E, uint64_t N,
                                  uint64_t Kd);

// Host: block-scale maps (no swizzle, boxes 16 bytes wide): a [rows, cols]
// byte tensor with box_rows rows per box, and the weights' [E, N, cols]
// scales with 128-row boxes (silu: 64 gate rows then the matching 64 up
// rows, as the weight tile).
bool make_tma_map_scales(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows);
bool make_tma_map_weight_scales(CUtensorMap* m, const void* base, bool silu, uint64_t E,
                                uint64_t N, uint64_t cols);

// Host: the weight map of a [E, N, Kd] tensor (see Maps::w): boxes of `kc`
// K chunks when Kd % 128 == 0 (weights_stage_box), else of one chunk;
// `silu`: the gate/up view of w13 (N = 2I).
inline bool weights_stage_box(uint64_t Kd) { return Kd % BK == 0; }
bool make_tma_map_weights(CUtensorMap* m, const void* base, bool silu, uint64_t E, uint64_t N,
                          uint64_t Kd, uint32_t kc);

}  // namespace gemm_common
}  // namespace moe
