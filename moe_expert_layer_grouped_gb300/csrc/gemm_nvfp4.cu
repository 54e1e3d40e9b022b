// The grouped GEMM in NVFP4, the FP4 format the pages deploy DeepSeek-R1 in
// ("[1/2] sgl-kernel: Fuse routed scaling factor into select_experts",
// sglang #8364, Motivation and Highlights: modelopt_fp4,
// ModelOptNvFp4FusedMoEMethod): E2M1 elements, one E4M3 scale per 16
// elements along K for every row of both operands, one fp32 global scale per
// tensor (ga for the activations, gb[e] per expert for the weights).
//   C[r,n] = ga * gb[e] * sum_k a[r,k] sa[r,k/16] * b[e,n,k] sb[e,n,k/16]
// with the block-scaled 5th-generation tensor-core MMA
// (tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X, K = 64 per
// instruction) and the same epilogues as the FP8 kernel (bf16 out, or
// SiLU(gate)*up with gate rows [j0, j0+64) and up rows [I+j0, I+j0+64) in one
// 128-row tile).
//
// Layouts: A [M, Kd/2] and B [E, N, Kd/2] bytes, two E2M1 codes per byte
// (element 2j in the low nibble), K-major; sa [M, Kd/16], sb [E, N, Kd/16]
// E4M3 codes. Kd % 256 == 0, so a 128-byte K chunk (256 elements) is whole.
//
// Design (one persistent CTA per SM, 320 threads, single-CTA MMAs):
//   warp 0      TMA producer, one or two K chunks per stage: the tile's 128
//               weight rows (one box), their scales (2 KB per chunk, already
//               in copy order, see below), the token rows (64/32/16-row
//               boxes) and their scale bytes (row-major).
//   warps 6..9  token scales, one warp per 32-lane quadrant of tensor
//               memory: each writes the stage's token scales from registers
//               (tcgen05.st) into its quadrant in the layout the MMA reads
//               (lane i, column 4j + c: the four scales of MMA step j of token
//               row i + 32c, the same in every quadrant) and signals the MMA
//               thread.
//               Lane 0 of warp 6 also copies the stage's four weight-scale
//               blocks (tcgen05.cp.32x128b.warpx4; block j: bytes of row
//               m0 + 32*m1 at offset 16*m0 + 4*m1, replicated into the four
//               quadrants), its commit being the last arrival the MMA thread
//               waits for.
//   warp 1      MMA: lane 0 issues the four MMAs of the chunk, each reading
//               its scales from four tensor-memory columns.
// Token scales go from registers to tensor memory rather than through a
// rearranged shared-memory block copied by tcgen05.cp: generic-proxy stores
// followed by a tcgen05.cp of the same bytes cost about 40 % of the decode
// w13 time in an earlier version.
//   warps 2..5  epilogue as in the FP8 kernel, dequantising by ga * gb[e].
// The weights' scales are arranged once, when the layer is set up
// (moe_nvfp4_arrange_scales): for expert e, weight tile nb (its 128 rows in
// the kernel's row order) and K chunk c, 2 KB holding the four blocks of the
// chunk's MMA steps, so a stage loads them with one bulk copy.
// Tensor memory: two accumulators of 128 columns (token tiles <= 128), then
// per pipeline stage 16 columns of weight scales and 16 of token scales,
// released with the stage.
// Every pipeline wait is bounded (2 s); on timeout the CTA sets the device
// error word, lets its in-flight copies and MMAs land, frees its tensor
// memory and exits.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace gemm_common;

constexpr int FT = 320;  // 10 warps: producer, MMA, 4 epilogue, 4 token scales
constexpr int SCALE_WARP0 = 6;
constexpr int SFROW = 16;      // scale bytes per row per 128-byte K chunk
constexpr uint32_t F_SFCHUNK = 32;  // scale columns per K chunk: 16 for the weights, 16 tokens
constexpr uint32_t F_TMEM = 512;
// Tile width FBN (tokens, MMA N), pipeline depth FSTAGES and K chunks per
// stage FKC per launch: few tokens per expert (decode) 64 tokens x 3 stages
// of 2 chunks, the weight stream's bytes in flight being what bounds it;
// otherwise 128 x 2 stages of 2 chunks (many tokens per expert go to the
// 256-row kernel of gemm_nvfp4_wide.cu whenever the weight rows split into
// 256-row tiles); one chunk per stage (6 / 5 stages) when the chunk count is
// odd. Tensor memory: two FBN-column accumulators, then FSTAGES x FKC x 32
// scale columns.

struct FMaps {
  CUtensorMap w;          // weights, one 128-byte chunk of 128 rows per box
  CUtensorMap x[NXBOX];   // token rows, boxes of 64 >> i rows
  CUtensorMap sx[NXBOX];  // token scales, 16 bytes x (64 >> i) rows
};

template <bool SILU, int FBN, int FSTAGES, int FKC>
struct FSmem {
  uint8_t w[FSTAGES][FKC * W_BYTES];       // FKC K chunks of the tile's weight rows (one box)
  uint8_t x[FSTAGES][FKC][FBN * BK];
  uint8_t sx[FSTAGES][FKC][FBN * SFROW];   // token scales, row-major as loaded
  uint32_t atom_a[FSTAGES][FKC * 4][128];  // weight scales: tcgen05.cp sources, one per MMA step
  float xchg[SILU ? 2 : 1][2][32 * 32];
  uint16_t stage_out[4][32 * 32];
  uint64_t full[FSTAGES];
  uint64_t sready[FSTAGES];  // the stage's token scales are in tensor memory
  uint64_t empty[FSTAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t sdrain;  // the weight-scale copies, before the teardown
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int never;
  int thr_sum[FT];
  int tile_start[MAX_E + 1];
  int offs[MAX_E + 1];
};

struct FParams {
  float ga;
  const float* gb;
  const uint8_t* sba;  // arranged weight scales [E][NB][KB][2048]
  const int32_t* offsets;
  void* C;
  int* err;
  int M, N, Kd, E, I, NB, KB;
  int stream_weights;
  int early_table;
  int stall_stage;  // failure test: CTA 0 never loads its stage with this index (-1: none)
};

template <bool SILU, int FBN, int FSTAGES, int FKC>
__global__ void __launch_bounds__(FT, 1)
    grouped_gemm_nvfp4_kernel(const __grid_constant__ FMaps maps, const FParams p) {
  constexpr uint32_t F_ACC = FBN;              // TMEM columns per accumulator
  constexpr uint32_t F_SF0 = 2 * F_ACC;        // first scale column
  constexpr uint32_t F_SFSTAGE = FKC * F_SFCHUNK;  // scale columns per stage
  static_assert(F_SF0 + FSTAGES * F_SFSTAGE <= F_TMEM, "tensor memory budget");
  using S = FSmem<SILU, FBN, FSTAGES, FKC>;
  extern __shared__ uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;
  const int KS = p.KB / FKC;  // FKC K chunks per stage (KB % FKC == 0)

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&maps.w);
    for (int i = 0; i < NXBOX; ++i) {
      ptx::prefetch_tensormap(&maps.x[i]);
      ptx::prefetch_tensormap(&maps.sx[i]);
    }
    for (int s = 0; s < FSTAGES; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      // one arrival per scale warp and the commit of the weight-scale copies
      ptx::mbar_init(&sm.sready[s], 5);
      ptx::mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sm.tfull[b], 1);
      ptx::mbar_init(&sm.tempty[b], 128);
    }
    ptx::mbar_init(&sm.drain, 1);
    ptx::mbar_init(&sm.sdrain, 1);
    sm.abort = 0;
    sm.never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, F_TMEM);
    ptx::tmem_relinquish();
  }
  if (!p.early_table) chain_entry();
  build_tile_table<FBN, FT>(sm, p.offsets, E, p.M, p.NB, p.err, tid);
  if (p.early_table) chain_entry();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int total = sm.total_tiles;

  uint32_t armed = 0, armed_par = 0;
  if (warp == 0) {
    // ======================= TMA producer ===================================
    if (lane == 0) {
      const uint64_t pol_w = p.stream_weights ? ptx::policy_evict_first() : ptx::policy_evict_normal();
      const uint64_t pol_w1 = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      uint32_t s = 0, ph = 0;
      int gstage = 0;  // stages issued by this CTA
      bool ok = true;
      for (int g = blockIdx.x; ok && g < total; g += gridDim.x) {
        const TileInfo<FBN> t = decode_tile<FBN>(sm, E, p.NB, g);
        const int rows = (t.ntok + 15) & ~15;
        const uint32_t bytes = FKC * (W_BYTES + 4 * 512 + (uint32_t)rows * (BK + SFROW));
        const uint8_t* sba = p.sba + (((int64_t)t.e * p.NB + t.nb) * p.KB) * 2048;
        const int y0 = t.e * p.N + t.nb * BM;  // bf16 epilogue: first weight row
        const uint64_t pw = t.nch == 1 ? pol_w1 : pol_w;
        for (int ks = 0; ks < KS; ++ks) {
          if (!ptx::mbar_wait(&sm.empty[s], ph ^ 1u, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&sm.full[s], bytes);
          armed |= 1u << s;
          armed_par = (armed_par & ~(1u << s)) | (ph << s);
          // failure test: the stage is armed but its bytes never come, so the
          // bounded waits run out
          if (blockIdx.x == 0 && gstage++ == p.stall_stage) {
            if (++s == FSTAGES) {
              s = 0;
              ph ^= 1u;
            }
            continue;
          }
          const int c0 = ks * FKC;  // the stage's first K chunk
          if (SILU)
            ptx::tma_load_5d(sm.w[s], &maps.w, &sm.full[s], 0, t.nb * 64, 0, c0, t.e, pw);
          else
            ptx::tma_load_3d(sm.w[s], &maps.w, &sm.full[s], 0, y0, c0, pw);
          ptx::bulk_load(sm.atom_a[s], sba + (int64_t)c0 * 2048, FKC * 4 * 512, &sm.full[s], pw);
#pragma unroll
          for (int kc = 0; kc < FKC; ++kc) {
            int r = 0;
#pragma unroll
            for (int i = 0; i < NXBOX; ++i) {
              const int box = 64 >> i;
              while (rows - r >= box) {
                ptx::tma_load_2d(sm.x[s][kc] + r * BK, &maps.x[i], &sm.full[s], (c0 + kc) * BK,
                                 t.tok0 + r, pol_x);
                ptx::tma_load_2d(sm.sx[s][kc] + r * SFROW, &maps.sx[i], &sm.full[s],
                                 (c0 + kc) * SFROW, t.tok0 + r, pol_x);
                r += box;
              }
            }
          }
          if (++s == FSTAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =====================================
    if (lane == 0) {
      uint32_t s = 0, ph = 0;
      bool ok = true, issued = false;
      int iter = 0;
      for (int g = blockIdx.x; ok && g < total; g += gridDim.x, ++iter) {
        const TileInfo<FBN> t = decode_tile<FBN>(sm, E, p.NB, g);
        const int n_mma = (t.ntok + 15) & ~15;
        const uint32_t idesc = ptx::idesc_nvfp4(BM, n_mma);
        const int b = iter & 1;
        const uint32_t tph = (iter >> 1) & 1;
        if (!ptx::mbar_wait(&sm.tempty[b], tph ^ 1u, &sm.abort, WAIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)b * F_ACC;
        for (int ks = 0; ks < KS; ++ks) {
          if (!ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS) ||
              !ptx::mbar_wait(&sm.sready[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int kc = 0; kc < FKC; ++kc) {
            const uint32_t sfa = tmem + F_SF0 + (uint32_t)s * F_SFSTAGE + kc * F_SFCHUNK;
            const uint32_t sfb = sfa + 16;
            const uint32_t a0 = ptx::smem_u32(sm.w[s]) + kc * W_BYTES;
            const uint32_t b0 = ptx::smem_u32(sm.x[s][kc]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              ptx::mma_nvfp4(d, ptx::sdesc_sw128(a0 + j * 32), ptx::sdesc_sw128(b0 + j * 32),
                             idesc, sfa + 4 * j, sfb + 4 * j, (ks | kc | j) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(&sm.empty[s]);
          issued = true;
          if (++s == FSTAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&sm.tfull[b]);
      }
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        if (issued) {
          ptx::mma_commit(&sm.drain);
          ptx::mbar_wait(&sm.drain, 0, &sm.never, DRAIN_NS);
        }
      }
    }
  } else if (warp >= SCALE_WARP0) {
    // ======================= token scales (warps 6..9) ======================
    // lane i of this warp's quadrant, register 4j + c: the four scales of MMA
    // step j of token row i + 32c (rows past the tile: zero)
    const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t s = 0, ph = 0;
    bool ok = true;
    for (int g = blockIdx.x; ok && g < total; g += gridDim.x) {
      for (int ks = 0; ks < KS; ++ks) {
        if (!__all_sync(kFull, ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS))) {
          ok = false;
          break;
        }
        if (warp == SCALE_WARP0 && lane == 0) {
          // the weights' scale blocks into the stage's columns, ahead of the
          // MMAs; the commit is the fifth arrival on sready
          ptx::tc_fence_after();
#pragma unroll
          for (int kc = 0; kc < FKC; ++kc) {
            const uint32_t sfa = tmem + F_SF0 + (uint32_t)s * F_SFSTAGE + kc * F_SFCHUNK;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              ptx::tmem_cp_32x128b_x4(sfa + 4 * j,
                                      ptx::sdesc_rows16(ptx::smem_u32(sm.atom_a[s][kc * 4 + j])));
          }
          ptx::mma_commit(&sm.sready[s]);
        }
#pragma unroll
        for (int kc = 0; kc < FKC; ++kc) {
          uint32_t r[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int row = lane + 32 * c;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row < FBN) v = *reinterpret_cast<const uint4*>(sm.sx[s][kc] + row * SFROW);
            r[c] = v.x;
            r[4 + c] = v.y;
            r[8 + c] = v.z;
            r[12 + c] = v.w;
          }
          ptx::tmem_st_32x32b_x16(tq + F_SF0 + (uint32_t)s * F_SFSTAGE + kc * F_SFCHUNK + 16, r);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.sready[s]);
        if (++s == FSTAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (lane == 0) {
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
      }
      // the copies this thread issued land before the tensor memory is freed
      // (at once when the MMA thread has waited for them all)
      if (warp == SCALE_WARP0) {
        ptx::mma_commit(&sm.sdrain);
        ptx::mbar_wait(&sm.sdrain, 0, &sm.never, DRAIN_NS);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ======================= epilogue (warps 2..5) ==========================
    const int q = warp & 3;
    int iter = 0;
    for (int g = blockIdx.x; g < total; g += gridDim.x, ++iter) {
      const TileInfo<FBN> t = decode_tile<FBN>(sm, E, p.NB, g);
      const int b = iter & 1;
      const uint32_t tph = (iter >> 1) & 1;
      bool ok = ptx::mbar_wait(&sm.tfull[b], tph, &sm.abort, WAIT_NS);
      ok = __all_sync(kFull, ok);
      if (SILU) ok = !bar_red_or(1 + (q & 1), 64, !ok);
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * F_ACC;
      const int nchunk = (t.ntok + 31) >> 5;
      const float scale = p.ga * __ldg(p.gb + t.e);  // both global scales
      uint16_t* ost = sm.stage_out[q];
      if (SILU) {
        const int I = p.I;
        const int pair = q & 1;
        const bool holds_gate = q < 2;
        __nv_bfloat16* hbase = reinterpret_cast<__nv_bfloat16*>(p.C);
        const int mine0 = holds_gate ? 0 : 16;
        const int jrow = t.nb * 64 + pair * 32;
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tbase, v);
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          ptx::tmem_ld_wait();
          ptx::reg_fence(v);
          float* give = sm.xchg[pair][c & 1] + (holds_gate ? 16 * 32 : 0);
          const float* take = sm.xchg[pair][c & 1] + (holds_gate ? 0 : 16 * 32);
          float own_v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float lo = __uint_as_float(v[i]), hi = __uint_as_float(v[16 + i]);
            own_v[i] = holds_gate ? lo : hi;
            give[i * 32 + lane] = holds_gate ? hi : lo;
          }
          if (c + 1 < nchunk) ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * 32, v);
          bar_sync_named(1 + pair, 64);
          const int tk0 = c * 32 + mine0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float other = take[i * 32 + lane];
            const float gv = (holds_gate ? own_v[i] : other) * scale;
            const float uv = (holds_gate ? other : own_v[i]) * scale;
            // the result is rounded to bf16, so a fast divide is well inside it
            ost[i * 32 + lane] = __bfloat16_as_ushort(
                __float2bfloat16_rn(__fdividef(gv, 1.0f + __expf(-gv)) * uv));
          }
          __syncwarp();
          if (jrow < I) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int r = k * 8 + (lane >> 2);
              if (tk0 + r < t.ntok)
                *reinterpret_cast<uint4*>(hbase + (int64_t)(t.tok0 + tk0 + r) * I + jrow +
                                          (lane & 3) * 8) =
                    *reinterpret_cast<const uint4*>(ost + r * 32 + (lane & 3) * 8);
            }
          }
          __syncwarp();
        }
        bar_sync_named(1 + pair, 64);
      } else {
        const int N = p.N;
        const int ncol0 = t.nb * BM + q * 32;
        __nv_bfloat16* cbase = reinterpret_cast<__nv_bfloat16*>(p.C);
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tbase, v);
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          ptx::tmem_ld_wait();
          ptx::reg_fence(v);
          float f[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
          if (c + 1 < nchunk) ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * 32, v);
          const int tk0 = c * 32;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            ost[i * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(f[i] * scale));
          __syncwarp();
          if (ncol0 < N) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int r = k * 8 + (lane >> 2);
              if (tk0 + r < t.ntok)
                *reinterpret_cast<uint4*>(cbase + (int64_t)(t.tok0 + tk0 + r) * N + ncol0 +
                                          (lane & 3) * 8) =
                    *reinterpret_cast<const uint4*>(ost + r * 32 + (lane & 3) * 8);
            }
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.tempty[b]);
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *reinterpret_cast<volatile int*>(&sm.abort))
    for (int i = 0; i < FSTAGES; ++i)
      if ((armed >> i) & 1u)
        ptx::mbar_wait(&sm.full[i], (armed_par >> i) & 1u, &sm.never, DRAIN_NS);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, F_TMEM);
  }
}

template <bool SILU, int FBN, int FSTAGES, int FKC>
cudaError_t launch_f(const FMaps& maps, const FParams& p, int M, int E, cudaStream_t st,
                     bool pdl) {
  constexpr size_t smem = sizeof(FSmem<SILU, FBN, FSTAGES, FKC>) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = grouped_gemm_nvfp4_kernel<SILU, FBN, FSTAGES, FKC>;
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
  const long long upper = ((long long)(M + FBN - 1) / FBN + E) * p.NB;
  const int grid = (int)std::max<long long>(1, std::min<long long>(sm_count(), upper));
  return launch_kernel(kern, dim3(grid), dim3(FT), smem, st, pdl, maps, p);
}

// Weight scales sb [E][N][Kd/16] -> the kernel's copy order: for expert e,
// weight tile nb, K chunk c, MMA step j: 512 bytes, byte 16*(m%32) +
// 4*(m/32) + b = scale 4j+b of chunk c of the tile's row m (SiLU tiles: rows
// m < 64 are gate rows 64nb+m, the rest up rows I+64nb+m-64). One thread
// per (e, nb, c, m).
__global__ void arrange_scales_kernel(const uint8_t* __restrict__ sb, int E, int N, int KB,
                                      int silu, uint8_t* __restrict__ out) {
  const int NB = silu ? N / 2 / 64 : N / BM;
  const int64_t n = (int64_t)E * NB * KB * BM;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(i % BM);
    const int64_t tc = i / BM;  // (e, nb, c)
    const int c = (int)(tc % KB);
    const int64_t enb = tc / KB;
    const int nb = (int)(enb % NB);
    const int e = (int)(enb / NB);
    const int I = N / 2;
    const int row = silu ? (m < 64 ? nb * 64 + m : I + nb * 64 + (m - 64)) : nb * BM + m;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(
        sb + ((int64_t)e * N + row) * (KB * 16) + (int64_t)c * 16);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + tc * 2048);
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j * 128 + (m % 32) * 4 + (m / 32)] = __ldg(src + j);
  }
}

}  // namespace

cudaError_t launch_nvfp4_arrange_scales(const uint8_t* sb, int E, int N, int Kd, int epilogue,
                                        uint8_t* out, cudaStream_t st) {
  const bool silu = epilogue == MOE_EPI_SILU_MUL;
  const int KB = Kd / 256;
  const int NB = silu ? N / 2 / 64 : N / BM;
  const int64_t n = (int64_t)E * NB * KB * BM;
  if (n == 0) return cudaSuccess;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 32);
  arrange_scales_kernel<<<blocks, 256, 0, st>>>(sb, E, N, KB, silu ? 1 : 0, out);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm_nvfp4(const void* A, const uint8_t* sfa, float ga, const void* B,
                                      const uint8_t* sfb, const float* gb,
                                      const int32_t* offsets, int M, int N, int Kd, int E,
                                      int epilogue, void* C, int* err, cudaStream_t st, bool pdl,
                                      bool early_table, int stall_stage) {
  if (M == 0) return cudaSuccess;
  // many rows per expert: 256 weight rows per CTA (gemm_nvfp4_wide.cu), which
  // stages each token row half as often
  if (gemm_nvfp4_wide_applies(M, N, Kd, E, epilogue))
    return launch_grouped_gemm_nvfp4_wide(A, sfa, ga, B, sfb, gb, offsets, M, N, Kd, E, epilogue,
                                          C, err, st, pdl, early_table, stall_stage);
  const bool silu = (epilogue == MOE_EPI_SILU_MUL);
  const uint64_t kb = (uint64_t)Kd / 2;   // bytes of a row
  const uint64_t sc = (uint64_t)Kd / 16;  // scale bytes of a row
  // two K chunks per stage (256 contiguous bytes of every weight row, half the
  // barrier round trips per byte) when the chunk count is even
  const bool many = gemm_many_rows(M, E);
  const int fkc = ((Kd / 256) % 2 == 0) ? 2 : 1;
  FMaps maps;
  if (!make_tma_map_weights(&maps.w, B, silu, (uint64_t)E, (uint64_t)N, kb, (uint32_t)fkc))
    return cudaErrorNotSupported;
  for (int i = 0; i < NXBOX; ++i)
    if (!make_tma_map_u8(&maps.x[i], A, (uint64_t)M, kb, 64u >> i) ||
        !make_tma_map_scales(&maps.sx[i], sfa, (uint64_t)M, sc, 64u >> i))
      return cudaErrorNotSupported;
  FParams p;
  p.ga = ga;
  p.gb = gb;
  p.sba = sfb;
  p.offsets = offsets;
  p.C = C;
  p.err = err;
  p.M = M;
  p.N = N;
  p.Kd = Kd;
  p.E = E;
  p.I = N / 2;
  p.NB = silu ? p.I / 64 : N / BM;
  p.KB = Kd / 256;
  p.stream_weights = many ? 0 : 1;
  p.early_table = early_table ? 1 : 0;
  p.stall_stage = stall_stage;
  if (!many && fkc == 2)
    return silu ? launch_f<true, 64, 3, 2>(maps, p, M, E, st, pdl)
                : launch_f<false, 64, 3, 2>(maps, p, M, E, st, pdl);
  if (!many)
    return silu ? launch_f<true, 64, 6, 1>(maps, p, M, E, st, pdl)
                : launch_f<false, 64, 6, 1>(maps, p, M, E, st, pdl);
  if (fkc == 2)
    return silu ? launch_f<true, 128, 2, 2>(maps, p, M, E, st, pdl)
                : launch_f<false, 128, 2, 2>(maps, p, M, E, st, pdl);
  return silu ? launch_f<true, 128, 5, 1>(maps, p, M, E, st, pdl)
              : launch_f<false, 128, 5, 1>(maps, p, M, E, st, pdl);
}

}  // namespace moe
