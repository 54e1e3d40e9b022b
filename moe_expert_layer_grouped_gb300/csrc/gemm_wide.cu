// The per-token FP8 grouped GEMM for long K (w13 at prefill, and w2 when the
// intermediate size is large) on CTA pairs with two accumulators per CTA.
//
// The pair kernel of gemm.cu gives each CTA 128 weight rows, so a pair tile
// of 256 weight rows x N tokens stages every token row once per 256 weight
// rows. Here each CTA holds 256 weight rows in two 128-row accumulators of
// the 2-SM MMA (tcgen05.mma.cta_group::2, M = 256 = 128 rows of each CTA,
// issued twice per K step on the same token operand). A pair tile covers 512
// weight rows, so the tokens are staged half as often: per K block a CTA
// stages 32 KB of weights and 16 KB of tokens for 16.8 MFLOP, against 32 KB
// for 8.4 MFLOP.
//
// SiLU*mul: a CTA's 256 rows are 128 gate rows, then the matching 128 up rows
// (one TMA box of the w13 view). So accumulator 0 holds gate j and
// accumulator 1 holds up j in the same TMEM lane, and an epilogue thread has
// both halves of its j without any exchange.
//
// The two accumulators fill the 512 TMEM columns (N <= 256 tokens each), so a
// tile's drain is not overlapped with the next tile's MMAs. The kernel is
// used only where K is long (at least 32 blocks of 128), which keeps the
// drain a small share of a tile.
//
// Roles (320 threads): warp 0 TMA producer, warp 1 the MMA issuer (the even
// CTA's lane 0 issues for both), warps 2-9 the epilogue (lane quadrant w % 4,
// two warps per quadrant on alternate token chunks, so a tile drains faster).
// Every wait is bounded: on timeout the CTA sets the device error word, lets
// its copies and MMAs land, frees its tensor memory and leaves.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace gemm_common;

constexpr int WEW = 8;               // epilogue warps: two per TMEM lane quadrant
constexpr int WT = 64 + 32 * WEW;
// K blocks per pipeline stage: 2 (two stages of 96 KB) measured slower than
// 1 (four of 48 KB): DeepSeek-V3 prefill w13 1.56 against 1.48 ms
constexpr int WKC = 1;
constexpr int WSTAGES = 4 / WKC;    // 192 KB of stages
constexpr int WROWS = 256;          // weight rows per CTA (two accumulators)
constexpr int WBN = 256;            // tokens per pair tile (MMA N), half per CTA
constexpr uint32_t WACC = 256;      // TMEM columns per accumulator
constexpr uint32_t WTMEM = 2 * WACC;

struct WSmem {
  uint8_t w[WSTAGES][WKC][WROWS * BK];      // this CTA's 256 weight rows, WKC K blocks
  uint8_t x[WSTAGES][WKC][(WBN / 2) * BK];  // this CTA's half of the tile's tokens
  uint16_t stage_out[WEW][32 * 32];    // per epilogue warp: bf16 [token][32 columns]
  uint64_t full[WSTAGES];              // only the even CTA's are armed and waited
  uint64_t empty[WSTAGES];
  uint64_t tfull;                      // the tile's accumulators are complete
  uint64_t tempty;                     // both CTAs' epilogues have drained them
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int never;
  int thr_sum[32];
  int tile_start[MAX_E + 1];
  int offs[MAX_E + 1];
};

struct WParams {
  const float* scale_a;
  const float* scale_b;
  const int32_t* offsets;
  void* C;
  int* err;
  int M, N, Kd, E, I, NBG, KB;
  int stream_weights;
  int early_table;
  int stall_stage;  // failure test: CTA 0 never loads its stage with this index (-1: none)
};

template <bool SILU>
__global__ void __launch_bounds__(WT, 1)
    grouped_gemm_wide_kernel(const __grid_constant__ Maps maps, const WParams p) {
  extern __shared__ uint8_t smem_raw[];
  WSmem& sm = *reinterpret_cast<WSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;
  const int KS = (p.KB + WKC - 1) / WKC;  // pipeline stages per tile

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&maps.w);
    for (int i = 0; i < NXBOX; ++i) ptx::prefetch_tensormap(&maps.x[i]);
    for (int s = 0; s < WSTAGES; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], 1);
    }
    ptx::mbar_init(&sm.tfull, 1);
    ptx::mbar_init(&sm.tempty, 2 * 32 * WEW);  // every epilogue thread of both CTAs
    ptx::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    sm.never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&sm.tmem_base, WTMEM);
    ptx::tmem_relinquish_pair();
  }
  const int rank = (int)ptx::cluster_ctarank();
  const int cluster = blockIdx.x / 2;
  const int nclusters = gridDim.x / 2;
  constexpr uint16_t kPair = 0x3;
  ptx::cluster_sync();  // the peer's barriers exist before any signal

  if (!p.early_table) chain_entry();
  build_tile_table<WBN, WT>(sm, p.offsets, E, p.M, p.NBG, p.err, tid);
  if (p.early_table) chain_entry();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int total = sm.total_tiles;

  uint32_t armed = 0, armed_par = 0;
  if (warp == 0) {
    // ======================= TMA producer ===================================
    const uint64_t pol_w = p.stream_weights ? ptx::policy_evict_first() : ptx::policy_evict_normal();
    const uint64_t pol_w1 = ptx::policy_evict_first();
    const uint64_t pol_x = ptx::policy_evict_last();
    uint32_t s = 0, ph = 0;
    int gstage = 0;  // stages issued by this CTA
    bool ok = true;
    for (int g = cluster; ok && g < total; g += nclusters) {
      const TileInfo<WBN> t = decode_tile<WBN>(sm, E, p.NBG, g);
      // token rows of the MMA: a multiple of 32, half in each CTA
      const int rows = (t.ntok + 31) & ~31;
      const int half = rows / 2;
      const uint32_t bytes = WKC * (uint32_t)(2 * WROWS + rows) * BK;  // both CTAs' loads
      const uint64_t pw = t.nch == 1 ? pol_w1 : pol_w;
      const int blk = t.nb * 2 + rank;       // this CTA's 256-row weight block
      const int jq = blk * 128;              // SiLU: its first j
      const int y0 = t.e * p.N + blk * WROWS;  // bf16: its first weight row
      for (int ks = 0; ks < KS; ++ks) {
        const bool got = ptx::mbar_wait(&sm.empty[s], ph ^ 1u, &sm.abort, WAIT_NS);
        if (!__all_sync(kFull, got)) {
          ok = false;
          break;
        }
        const uint32_t fb = ptx::map_to_rank(ptx::smem_u32(&sm.full[s]), 0);
        // failure test: the stage is armed but this CTA's bytes never come,
        // so the bounded waits run out
        const bool stall = blockIdx.x == 0 && gstage++ == p.stall_stage;
        if (lane == 0) {
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(&sm.full[s], bytes);
            armed |= 1u << s;
            armed_par = (armed_par & ~(1u << s)) | (ph << s);
          }
        }
        if (lane == 0 && !stall) {
          // the stage's WKC K blocks (past Kd: zero-filled, adding nothing)
          if (SILU)  // per K block 128 gate rows, then the matching 128 up rows
            ptx::tma_load_5d_pair(sm.w[s][0], &maps.w, fb, 0, jq, 0, ks * WKC, t.e, pw);
          else
            ptx::tma_load_3d_pair(sm.w[s][0], &maps.w, fb, 0, y0, ks * WKC, pw);
#pragma unroll
          for (int kc = 0; kc < WKC; ++kc) {
            int r = 0;
#pragma unroll
            for (int i = 0; i < NXBOX; ++i) {
              const int box = 64 >> i;
              while (half - r >= box) {
                ptx::tma_load_2d_pair(sm.x[s][kc] + r * BK, &maps.x[i], fb, (ks * WKC + kc) * BK,
                                      t.tok0 + rank * half + r, pol_x);
                r += box;
              }
            }
          }
        }
        if (++s == WSTAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      sm.abort = 1;
      flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =====================================
    if (lane == 0 && rank == 0) {
      uint32_t s = 0, ph = 0;
      bool ok = true, issued = false;
      int iter = 0;
      for (int g = cluster; ok && g < total; g += nclusters, ++iter) {
        const TileInfo<WBN> t = decode_tile<WBN>(sm, E, p.NBG, g);
        const int n_mma = (t.ntok + 31) & ~31;
        const uint32_t idesc = ptx::idesc_e4m3_f32(256, n_mma);
        // both accumulators drained by both CTAs' epilogues
        if (!ptx::mbar_wait(&sm.tempty, (uint32_t)(iter & 1) ^ 1u, &sm.abort, WAIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int ks = 0; ks < KS; ++ks) {
          if (!ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int kc = 0; kc < WKC; ++kc) {
            const uint32_t b0 = ptx::smem_u32(sm.x[s][kc]);
#pragma unroll
            for (int acc = 0; acc < 2; ++acc) {
              const uint32_t a0 = ptx::smem_u32(sm.w[s][kc]) + (uint32_t)acc * 128 * BK;
#pragma unroll
              for (int kk = 0; kk < BK / 32; ++kk)
                ptx::mma_e4m3_pair(tmem + (uint32_t)acc * WACC, ptx::sdesc_sw128(a0 + kk * 32),
                                   ptx::sdesc_sw128(b0 + kk * 32), idesc,
                                   (ks | kc | kk) != 0 ? 1u : 0u);
            }
          }
          issued = true;
          ptx::mma_commit_pair_mcast(&sm.empty[s], kPair);  // frees the stage in both CTAs
          if (++s == WSTAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_mcast(&sm.tfull, kPair);  // both CTAs' epilogues
      }
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        if (issued) {
          ptx::mma_commit_pair_mcast(&sm.drain, 0x1);
          ptx::mbar_wait(&sm.drain, 0, &sm.never, DRAIN_NS);
        }
      }
    }
  } else {
    // ======================= epilogue (warps 2..) ===========================
    // warp w reads lane quadrant w % 4; the two warps of a quadrant take the
    // even and the odd 32-token chunks
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int par = (warp - 2) / 4;
    int iter = 0;
    for (int g = cluster; g < total; g += nclusters, ++iter) {
      const TileInfo<WBN> t = decode_tile<WBN>(sm, E, p.NBG, g);
      bool ok = ptx::mbar_wait(&sm.tfull, (uint32_t)(iter & 1), &sm.abort, WAIT_NS);
      if (!__all_sync(kFull, ok)) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
      const int nchunk = (t.ntok + 31) >> 5;
      const int64_t e = t.e;
      const int blk = t.nb * 2 + rank;
      uint16_t* ost = sm.stage_out[warp - 2];
      if (SILU) {
        const int I = p.I;
        const int jrow = blk * 128 + q * 32;  // first j of this warp's 32
        const int j = jrow + lane;
        const float sg = __ldg(p.scale_b + e * p.N + j);
        const float su = __ldg(p.scale_b + e * p.N + I + j);
        __nv_bfloat16* hbase = reinterpret_cast<__nv_bfloat16*>(p.C);
#pragma unroll 1
        for (int c = par; c < nchunk; c += WEW / 4) {
          uint32_t gv[32], uv[32];
          ptx::tmem_ld_32x32b_x32(tq + c * 32, gv);
          ptx::tmem_ld_32x32b_x32(tq + WACC + c * 32, uv);
          ptx::tmem_ld_wait();
          ptx::reg_fence(gv);
          ptx::reg_fence(uv);
          const int tk0 = c * 32;
          const float sa_l = (tk0 + lane < t.ntok) ? __ldg(p.scale_a + t.tok0 + tk0 + lane) : 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float sa = __shfl_sync(kFull, sa_l, i);
            const float gg = __uint_as_float(gv[i]) * sa * sg;
            const float uu = __uint_as_float(uv[i]) * sa * su;
            // silu(g) * u, rounded to bf16: a fast divide (2 ulp) is well
            // inside that precision
            ost[i * 32 + lane] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__fdividef(gg, 1.0f + __expf(-gg)) * uu));
          }
          __syncwarp();
          // 32 tokens x 32 j: four lanes per token row, 16 bytes each
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int r = k * 8 + (lane >> 2);
            if (tk0 + r < t.ntok)
              *reinterpret_cast<uint4*>(hbase + (int64_t)(t.tok0 + tk0 + r) * I + jrow +
                                        (lane & 3) * 8) =
                  *reinterpret_cast<const uint4*>(ost + r * 32 + (lane & 3) * 8);
          }
          __syncwarp();
        }
      } else {
        const int N = p.N;
        __nv_bfloat16* cbase = reinterpret_cast<__nv_bfloat16*>(p.C);
#pragma unroll 1
        for (int acc = 0; acc < 2; ++acc) {
          const int ncol0 = blk * WROWS + acc * 128 + q * 32;  // first column of this warp's 32
          const float sb = __ldg(p.scale_b + e * N + ncol0 + lane);
#pragma unroll 1
          for (int c = par; c < nchunk; c += WEW / 4) {
            uint32_t v[32];
            ptx::tmem_ld_sync_x32(tq + (uint32_t)acc * WACC + c * 32, v);
            const int tk0 = c * 32;
            const float sa_l =
                (tk0 + lane < t.ntok) ? __ldg(p.scale_a + t.tok0 + tk0 + lane) : 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float sa = __shfl_sync(kFull, sa_l, i);
              ost[i * 32 + lane] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i]) * sa * sb));
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int r = k * 8 + (lane >> 2);
              if (tk0 + r < t.ntok)
                *reinterpret_cast<uint4*>(cbase + (int64_t)(t.tok0 + tk0 + r) * N + ncol0 +
                                          (lane & 3) * 8) =
                    *reinterpret_cast<const uint4*>(ost + r * 32 + (lane & 3) * 8);
            }
            __syncwarp();
          }
        }
      }
      ptx::tc_fence_before();
      if (rank != 0)
        ptx::mbar_arrive_cluster(ptx::map_to_rank(ptx::smem_u32(&sm.tempty), 0));
      else
        ptx::mbar_arrive(&sm.tempty);
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *reinterpret_cast<volatile int*>(&sm.abort))
    for (int i = 0; i < WSTAGES; ++i)
      if ((armed >> i) & 1u)
        ptx::mbar_wait(&sm.full[i], (armed_par >> i) & 1u, &sm.never, DRAIN_NS);
  // both CTAs are done with the shared accumulators before they are freed, and
  // neither leaves while the other may still signal its barriers
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, WTMEM);
  }
  ptx::cluster_sync();
}

template <bool SILU>
cudaError_t launch_wide_cfg(const Maps& maps, const WParams& p, int M, int E, cudaStream_t st,
                            bool pdl) {
  constexpr size_t smem = sizeof(WSmem) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = grouped_gemm_wide_kernel<SILU>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 64 || !attr_set[dev]) {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (dev < 64) attr_set[dev] = true;
    }
  }
  const long long upper = ((long long)(M + WBN - 1) / WBN + E) * p.NBG * 2;
  int grid = (int)std::min<long long>(sm_count(), upper);
  grid = std::max(2, grid / 2 * 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(WT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  // a persistent grid of pairs must be co-resident
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) == cudaSuccess && nclusters > 0)
    cfg.gridDim = dim3(std::min(grid, nclusters * 2));
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

}  // namespace

bool gemm_wide_applies(int M, int N, int Kd, int E, int epilogue) {
  if (!gemm_many_rows(M, E) || Kd % BK != 0 || Kd / BK < 32) return false;
  return epilogue == MOE_EPI_SILU_MUL ? (N / 2) % 256 == 0 : N % 512 == 0;
}

cudaError_t launch_grouped_gemm_wide(const void* A, const float* scale_a, const void* B,
                                     const float* scale_b, const int32_t* offsets, int M, int N,
                                     int Kd, int E, int epilogue, void* C, int* err,
                                     cudaStream_t st, bool pdl, bool early_table,
                                     int stall_stage) {
  if (M == 0) return cudaSuccess;
  const bool silu = (epilogue == MOE_EPI_SILU_MUL);
  Maps maps;
  const bool wok =
      silu ? make_tma_map_weights_gateup(&maps.w, B, (uint64_t)E, (uint64_t)N, (uint64_t)Kd, 128,
                                         WKC)
           : make_tma_map_weights_rows(&maps.w, B, (uint64_t)E, (uint64_t)N, (uint64_t)Kd,
                                       (uint32_t)WROWS, WKC);
  if (!wok) return cudaErrorNotSupported;
  for (int i = 0; i < NXBOX; ++i)
    if (!make_tma_map_u8(&maps.x[i], A, (uint64_t)M, (uint64_t)Kd, 64u >> i))
      return cudaErrorNotSupported;
  WParams p;
  p.scale_a = scale_a;
  p.scale_b = scale_b;
  p.offsets = offsets;
  p.C = C;
  p.err = err;
  p.M = M;
  p.N = N;
  p.Kd = Kd;
  p.E = E;
  p.I = N / 2;
  p.NBG = silu ? (N / 2) / 256 : N / 512;  // pair tiles of 512 weight rows per expert
  p.KB = Kd / BK;
  p.stream_weights = 0;
  p.early_table = early_table ? 1 : 0;
  p.stall_stage = stall_stage;
  return silu ? launch_wide_cfg<true>(maps, p, M, E, st, pdl)
              : launch_wide_cfg<false>(maps, p, M, E, st, pdl);
}

}  // namespace moe
