// The NVFP4 grouped GEMM for many tokens per expert (prefill) with 256 weight
// rows per CTA in two 128-row accumulators that share the token operand.
//
// The kernel of gemm_nvfp4.cu gives a CTA 128 weight rows x 128 tokens, so it
// stages 36 KB per 256 channels of K (16 KB of weight codes, 16 KB of token
// codes, 2 KB of scales each) for 8.4 MFLOP. At the FP4 tensor rate that
// stage would have to land every ~110 ns, and the operand feed into the SM,
// not the tensor pipe, sets the pace. Here a CTA holds 256 weight rows
// against the same 128 tokens: 54 KB per K chunk for 16.8 MFLOP, a third
// fewer staged bytes per FLOP.
//
// SiLU*mul: the 256 rows are 128 gate rows then the matching 128 up rows
// (one TMA box of the w13 view), so accumulator 0 holds gate j and
// accumulator 1 holds up j in the same tensor-memory lane and an epilogue
// thread has both halves of its j without an exchange.
//
// Scale factors. The weights' scales come arranged for the 128-row tiles of
// gemm_nvfp4.cu (per tile and K chunk, four 512-byte blocks, one per MMA
// step: byte 16*(m%32) + 4*(m/32) + b = scale b of the step for tile row m;
// SiLU tiles hold 64 gate rows then the matching 64 up rows). A wide tile is
// two of those tiles, loaded as two 2 KB bulk copies per K chunk. The MMA
// reads a 128-row operand's scales for step j from four tensor-memory
// columns, row r in lane r % 32 and column r / 32 of every lane quadrant
// (.scale_vec::4X; PTX ISA, tcgen05 "Block Scaling"). For a SiLU tile the
// gate accumulator's rows r < 64 are the first tile's gate rows and r >= 64
// the second's, so its column pairs come from different blocks and cannot be
// copied by tcgen05.cp as whole 16-byte lane rows. The scale warps therefore
// write every scale (weights and tokens) from registers with tcgen05.st.
//
// Roles (448 threads, one persistent CTA per SM):
//   warp 0      TMA producer: per K chunk the 256 weight rows (one box), the
//               two tiles' arranged scale blocks (two bulk copies), the token
//               rows (64/32/16-row boxes) and their scale bytes.
//   warp 1      MMA: lane 0 issues 2 x 4 MMAs per K chunk (K = 64 each).
//   warps 2..9  epilogue, lane quadrant warp % 4.
//   warps 10..13 scales: one warp per lane quadrant writes the stage's three
//               16-column scale groups (two weight halves, tokens) into its
//               quadrant and arrives on the stage's scale barrier. After a
//               tile's last stage it joins the tile's drain.
// A tile drains through three warps per lane quadrant (two epilogue warps and
// the scale warp), each taking every third 32-token item: the MMA thread
// cannot start the next tile before the drain ends, so the scale warps are
// not needed elsewhere meanwhile. The epilogue costs DeepSeek-V3's w2 about a
// quarter of its time (0.862 ms, 0.625 with the accumulators released
// unread, 0.752 without the output stores); the third warp per quadrant took
// it to 0.852 ms.
// Tensor memory: the two 128-column accumulators (one tile: its drain is not
// overlapped with the next tile's MMAs), then 48 scale columns per stage.
// Shared memory: four stages of 54 KB when the tile table (E + 1 entries
// twice, sized at launch) leaves room, i.e. up to ~470 experts, else three:
// DeepSeek-V3 prefill w13 1.283 -> 1.210 ms with the fourth stage, the drain
// then staged 8 tokens at a time to make room.
// Every wait is bounded (2 s); on timeout the CTA sets the device error word,
// lets its copies and MMAs land, frees its tensor memory and leaves.
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

constexpr int QEW = 8;                     // epilogue warps: two per lane quadrant
constexpr int QSW0 = 2 + QEW;              // first scale warp
constexpr int QT = 32 * (QSW0 + 4);        // 448 threads
constexpr int QDRAIN = QEW / 4 + 1;        // warps per lane quadrant that drain a tile
constexpr int QBN = 128;                   // tokens per tile (MMA N)
constexpr int QROWS = 256;                 // weight rows per tile (two accumulators)
constexpr int QSFROW = 16;                 // scale bytes per row per 128-byte K chunk
constexpr int QSUB = 8;                    // tokens per drain round (shared-memory tile)
constexpr uint32_t QACC = 128;             // tensor-memory columns per accumulator
constexpr uint32_t QSF0 = 2 * QACC;        // first scale column
constexpr uint32_t QSFSTAGE = 48;          // scale columns per stage: 16 + 16 weights, 16 tokens
constexpr uint32_t QTMEM = 512;
constexpr size_t QSMEM_MAX = 227 * 1024;

struct QMaps {
  CUtensorMap w;          // 256 weight rows of one 128-byte K chunk per box
  CUtensorMap x[NXBOX];   // token rows, boxes of 64 >> i rows
  CUtensorMap sx[NXBOX];  // token scales, 16 bytes x (64 >> i) rows
};

// The stage ring, 54 KB a stage, then the tile table (tile_start and offs,
// E + 1 entries each) after the struct, sized by the launch: four stages
// when they fit in the 227 KB with the table, else three.
template <int STG>
struct QSmem {
  static_assert(QSF0 + STG * QSFSTAGE <= QTMEM, "tensor memory budget");
  uint8_t w[STG][QROWS * BK];          // accumulator 0's rows, then accumulator 1's
  uint8_t x[STG][QBN * BK];
  uint8_t sx[STG][QBN * QSFROW];       // token scales, row-major as loaded
  uint4 sa[STG][2][4][32];             // the two tiles' arranged weight-scale blocks
  uint16_t stage_out[QEW + 4][QSUB * 32];  // per draining warp: bf16 [token][32 columns]
  uint64_t full[STG];
  uint64_t sready[STG];  // the stage's scales are in tensor memory
  uint64_t empty[STG];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int never;
  int thr_sum[32];
};

// The tile table's view for build_tile_table / decode_tile: the arrays live
// in the dynamic shared memory after the struct.
struct QTab {
  int* tile_start;
  int* offs;
  int* thr_sum;
  int& total_tiles;
};

struct QParams {
  float ga;
  const float* gb;
  const uint8_t* sba;  // arranged weight scales [E][NB][KB][2048] (128-row tiles)
  const int32_t* offsets;
  void* C;
  int* err;
  int M, N, Kd, E, I, NB, NBG, KB;
  int early_table;
  int stall_stage;  // failure test: CTA 0 never loads its stage with this index (-1: none)
};

// QSUB tokens x 32 columns from the warp's shared-memory tile to dst (row
// stride ld), tokens tk.. of tile t: four lanes per token row, 16 bytes each.
__device__ __forceinline__ void store_rows(uint16_t* ost, __nv_bfloat16* dst, int ld,
                                           const TileInfo<QBN>& t, int tk, int lane) {
  static_assert(QSUB * 4 == 32, "one 16-byte store per lane");
  __syncwarp();
  const int r = lane >> 2;
  if (tk + r < t.ntok)
    *reinterpret_cast<uint4*>(dst + (int64_t)(t.tok0 + tk + r) * ld + (lane & 3) * 8) =
        *reinterpret_cast<const uint4*>(ost + r * 32 + (lane & 3) * 8);
  __syncwarp();
}

// One warp's share of a tile's drain, in its lane quadrant q (TMEM lanes
// tq ..): the 32-token x 32-row items slot, slot + QDRAIN, ... of the tile.
// SiLU: item c = token chunk c of both accumulators (gate j and up j in the
// same lane), written as h columns; bf16: item it = accumulator it / nchunk,
// token chunk it % nchunk. Each item goes through the warp's shared-memory
// tile ost, QSUB tokens at a time, so that four lanes write a token's 64
// bytes in 16-byte stores.
template <bool SILU>
__device__ __forceinline__ void drain_items(const QParams& p, const TileInfo<QBN>& t,
                                            uint32_t tq, int q, int slot, uint16_t* ost,
                                            int lane) {
  const int nchunk = (t.ntok + 31) >> 5;
  const int items = SILU ? nchunk : 2 * nchunk;
  const float scale = p.ga * __ldg(p.gb + t.e);  // both global scales
#pragma unroll 1
  for (int it = slot; it < items; it += QDRAIN) {
    const int acc = SILU ? 0 : it / nchunk;
    const int c = it - acc * nchunk;
    const int tk0 = c * 32;
    __nv_bfloat16* dst;
    int ld;
    if (SILU) {
      uint32_t gv[32], uv[32];
      ptx::tmem_ld_32x32b_x32(tq + c * 32, gv);
      ptx::tmem_ld_32x32b_x32(tq + QACC + c * 32, uv);
      ptx::tmem_ld_wait();
      ptx::reg_fence(gv);
      ptx::reg_fence(uv);
      ld = p.I;
      dst = reinterpret_cast<__nv_bfloat16*>(p.C) + t.nb * 128 + q * 32;  // this warp's 32 j
      // QSUB tokens at a time through the shared-memory tile
#pragma unroll
      for (int i0 = 0; i0 < 32; i0 += QSUB) {
#pragma unroll
        for (int i = i0; i < i0 + QSUB; ++i) {
          const float gg = __uint_as_float(gv[i]) * scale;
          const float uu = __uint_as_float(uv[i]) * scale;
          // silu(g) * u, rounded to bf16: a fast divide is well inside it
          ost[(i - i0) * 32 + lane] =
              __bfloat16_as_ushort(__float2bfloat16_rn(__fdividef(gg, 1.0f + __expf(-gg)) * uu));
        }
        store_rows(ost, dst, ld, t, tk0 + i0, lane);
      }
    } else {
      uint32_t v[32];
      ptx::tmem_ld_sync_x32(tq + (uint32_t)acc * QACC + c * 32, v);
      ld = p.N;
      dst = reinterpret_cast<__nv_bfloat16*>(p.C) + t.nb * QROWS + acc * 128 + q * 32;
#pragma unroll
      for (int i0 = 0; i0 < 32; i0 += QSUB) {
#pragma unroll
        for (int i = i0; i < i0 + QSUB; ++i)
          ost[(i - i0) * 32 + lane] =
              __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i]) * scale));
        store_rows(ost, dst, ld, t, tk0 + i0, lane);
      }
    }
  }
}

template <bool SILU, int STG>
__global__ void __launch_bounds__(QT, 1)
    grouped_gemm_nvfp4_wide_kernel(const __grid_constant__ QMaps maps, const QParams p) {
  constexpr int QSTAGES = STG;
  extern __shared__ uint8_t smem_raw[];
  using S = QSmem<STG>;
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                ~static_cast<uintptr_t>(1023));
  int* const tab_mem = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(&sm) + sizeof(S));
  QTab tab{tab_mem, tab_mem + p.E + 1, sm.thr_sum, sm.total_tiles};
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;
  const int KS = p.KB;  // one K chunk per stage

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&maps.w);
    for (int i = 0; i < NXBOX; ++i) {
      ptx::prefetch_tensormap(&maps.x[i]);
      ptx::prefetch_tensormap(&maps.sx[i]);
    }
    for (int s = 0; s < QSTAGES; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.sready[s], 4);  // one arrival per scale warp
      ptx::mbar_init(&sm.empty[s], 1);
    }
    ptx::mbar_init(&sm.tfull, 1);
    ptx::mbar_init(&sm.tempty, 32 * (QEW + 4));  // every draining thread
    ptx::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    sm.never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, QTMEM);
    ptx::tmem_relinquish();
  }
  if (!p.early_table) chain_entry();
  build_tile_table<QBN, QT>(tab, p.offsets, E, p.M, p.NBG, p.err, tid);
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
      const uint64_t pol_w = ptx::policy_evict_normal();
      const uint64_t pol_w1 = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      uint32_t s = 0, ph = 0;
      int gstage = 0;  // stages issued by this CTA
      bool ok = true;
      for (int g = blockIdx.x; ok && g < total; g += gridDim.x) {
        const TileInfo<QBN> t = decode_tile<QBN>(tab, E, p.NBG, g);
        const int rows = (t.ntok + 15) & ~15;
        const uint32_t bytes = QROWS * BK + 2 * 2048 + (uint32_t)rows * (BK + QSFROW);
        // the two 128-row tiles' arranged scales, chunk 0
        const uint8_t* sb0 = p.sba + (((int64_t)t.e * p.NB + 2 * t.nb) * p.KB) * 2048;
        const uint8_t* sb1 = sb0 + (int64_t)p.KB * 2048;
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
            if (++s == QSTAGES) {
              s = 0;
              ph ^= 1u;
            }
            continue;
          }
          if (SILU)  // 128 gate rows from j = 128 nb, then the matching 128 up rows
            ptx::tma_load_5d(sm.w[s], &maps.w, &sm.full[s], 0, t.nb * 128, 0, ks, t.e, pw);
          else
            ptx::tma_load_3d(sm.w[s], &maps.w, &sm.full[s], 0, t.e * p.N + t.nb * QROWS, ks, pw);
          ptx::bulk_load(sm.sa[s][0], sb0 + (int64_t)ks * 2048, 2048, &sm.full[s], pw);
          ptx::bulk_load(sm.sa[s][1], sb1 + (int64_t)ks * 2048, 2048, &sm.full[s], pw);
          int r = 0;
#pragma unroll
          for (int i = 0; i < NXBOX; ++i) {
            const int box = 64 >> i;
            while (rows - r >= box) {
              ptx::tma_load_2d(sm.x[s] + r * BK, &maps.x[i], &sm.full[s], ks * BK, t.tok0 + r,
                               pol_x);
              ptx::tma_load_2d(sm.sx[s] + r * QSFROW, &maps.sx[i], &sm.full[s], ks * QSFROW,
                               t.tok0 + r, pol_x);
              r += box;
            }
          }
          if (++s == QSTAGES) {
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
        const TileInfo<QBN> t = decode_tile<QBN>(tab, E, p.NBG, g);
        const int n_mma = (t.ntok + 15) & ~15;
        const uint32_t idesc = ptx::idesc_nvfp4(BM, n_mma);
        if (!ptx::mbar_wait(&sm.tempty, (uint32_t)(iter & 1) ^ 1u, &sm.abort, WAIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int ks = 0; ks < KS; ++ks) {
          if (!ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS) ||
              !ptx::mbar_wait(&sm.sready[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sf = tmem + QSF0 + (uint32_t)s * QSFSTAGE;
          const uint32_t b0 = ptx::smem_u32(sm.x[s]);
#pragma unroll
          for (int acc = 0; acc < 2; ++acc) {
            const uint32_t a0 = ptx::smem_u32(sm.w[s]) + (uint32_t)acc * W_BYTES;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              ptx::mma_nvfp4(tmem + (uint32_t)acc * QACC, ptx::sdesc_sw128(a0 + j * 32),
                             ptx::sdesc_sw128(b0 + j * 32), idesc, sf + acc * 16 + 4 * j,
                             sf + 32 + 4 * j, (ks | j) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(&sm.empty[s]);
          issued = true;
          if (++s == QSTAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&sm.tfull);
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
  } else if (warp >= QSW0) {
    // ======================= scales (warps 10..13) ==========================
    // (and, after each tile's stages, a third of its drain)
    // Register 4j + c of lane i: the four scales of MMA step j of the
    // operand's row i + 32c. Weights, from the arranged blocks (lane i's
    // 16 bytes of block j: words c = 0..3 for tile rows i + 32c): bf16 tiles
    // map whole, SiLU accumulators take the gate (words 0, 1) or up (words
    // 2, 3) halves of both tiles. Tokens: row-major bytes of row i + 32c.
    const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t s = 0, ph = 0;
    bool ok = true;
    int iter = 0;
    for (int g = blockIdx.x; ok && g < total; g += gridDim.x, ++iter) {
      for (int ks = 0; ks < KS; ++ks) {
        if (!__all_sync(kFull, ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS))) {
          ok = false;
          break;
        }
        const uint32_t sf = tq + QSF0 + (uint32_t)s * QSFSTAGE;
        {
          uint32_t r0[16], r1[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 a = sm.sa[s][0][j][lane];
            const uint4 b = sm.sa[s][1][j][lane];
            if (SILU) {
              r0[4 * j + 0] = a.x;
              r0[4 * j + 1] = a.y;
              r0[4 * j + 2] = b.x;
              r0[4 * j + 3] = b.y;
              r1[4 * j + 0] = a.z;
              r1[4 * j + 1] = a.w;
              r1[4 * j + 2] = b.z;
              r1[4 * j + 3] = b.w;
            } else {
              r0[4 * j + 0] = a.x;
              r0[4 * j + 1] = a.y;
              r0[4 * j + 2] = a.z;
              r0[4 * j + 3] = a.w;
              r1[4 * j + 0] = b.x;
              r1[4 * j + 1] = b.y;
              r1[4 * j + 2] = b.z;
              r1[4 * j + 3] = b.w;
            }
          }
          ptx::tmem_st_32x32b_x16(sf, r0);
          ptx::tmem_st_32x32b_x16(sf + 16, r1);
        }
        {
          uint32_t r[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(sm.sx[s] + (lane + 32 * c) * QSFROW);
            r[c] = v.x;
            r[4 + c] = v.y;
            r[8 + c] = v.z;
            r[12 + c] = v.w;
          }
          ptx::tmem_st_32x32b_x16(sf + 32, r);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.sready[s]);
        if (++s == QSTAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      // then a third of the tile's drain: the MMA cannot start the next tile
      // before it ends, so the next stages' scales lose nothing by waiting
      const bool got = ptx::mbar_wait(&sm.tfull, (uint32_t)(iter & 1), &sm.abort, WAIT_NS);
      if (!__all_sync(kFull, got)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      drain_items<SILU>(p, decode_tile<QBN>(tab, E, p.NBG, g), tq, warp & 3, QDRAIN - 1,
                        sm.stage_out[warp - 2], lane);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.tempty);
    }
    if (!ok && lane == 0) {
      sm.abort = 1;
      flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
    }
  } else {
    // ======================= epilogue (warps 2..9) ==========================
    const int q = warp & 3;  // lane quadrant this warp may access
    const int par = (warp - 2) / 4;
    int iter = 0;
    for (int g = blockIdx.x; g < total; g += gridDim.x, ++iter) {
      const TileInfo<QBN> t = decode_tile<QBN>(tab, E, p.NBG, g);
      const bool ok = ptx::mbar_wait(&sm.tfull, (uint32_t)(iter & 1), &sm.abort, WAIT_NS);
      if (!__all_sync(kFull, ok)) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        break;
      }
      ptx::tc_fence_after();
      drain_items<SILU>(p, t, tmem + ((uint32_t)(q * 32) << 16), q, par, sm.stage_out[warp - 2],
                        lane);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.tempty);
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *reinterpret_cast<volatile int*>(&sm.abort))
    for (int i = 0; i < QSTAGES; ++i)
      if ((armed >> i) & 1u)
        ptx::mbar_wait(&sm.full[i], (armed_par >> i) & 1u, &sm.never, DRAIN_NS);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, QTMEM);
  }
}

template <int STG>
size_t q_smem_bytes(int E) {
  return sizeof(QSmem<STG>) + 2 * (size_t)(E + 1) * sizeof(int) + 1024;
}

template <bool SILU, int STG>
cudaError_t launch_q(const QMaps& maps, const QParams& p, int M, int E, cudaStream_t st,
                     bool pdl) {
  const size_t smem = q_smem_bytes<STG>(E);
  if (smem > QSMEM_MAX) return cudaErrorInvalidValue;
  auto kern = grouped_gemm_nvfp4_wide_kernel<SILU, STG>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 64 || !attr_set[dev]) {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QSMEM_MAX);
      if (e != cudaSuccess) return e;
      if (dev < 64) attr_set[dev] = true;
    }
  }
  const long long upper = ((long long)(M + QBN - 1) / QBN + E) * p.NBG;
  const int grid = (int)std::max<long long>(1, std::min<long long>(sm_count(), upper));
  return launch_kernel(kern, dim3(grid), dim3(QT), smem, st, pdl, maps, p);
}

}  // namespace

bool gemm_nvfp4_wide_applies(int M, int N, int Kd, int E, int epilogue) {
  if (!gemm_many_rows(M, E) || Kd % 256 != 0) return false;
  return epilogue == MOE_EPI_SILU_MUL ? (N / 2) % 128 == 0 : N % 256 == 0;
}

cudaError_t launch_grouped_gemm_nvfp4_wide(const void* A, const uint8_t* sfa, float ga,
                                           const void* B, const uint8_t* sfb, const float* gb,
                                           const int32_t* offsets, int M, int N, int Kd, int E,
                                           int epilogue, void* C, int* err, cudaStream_t st,
                                           bool pdl, bool early_table, int stall_stage) {
  if (M == 0) return cudaSuccess;
  const bool silu = (epilogue == MOE_EPI_SILU_MUL);
  const uint64_t kb = (uint64_t)Kd / 2;   // bytes of a row
  const uint64_t sc = (uint64_t)Kd / 16;  // scale bytes of a row
  QMaps maps;
  const bool wok = silu ? make_tma_map_weights_gateup(&maps.w, B, (uint64_t)E, (uint64_t)N, kb,
                                                      128, 1)
                        : make_tma_map_weights_rows(&maps.w, B, (uint64_t)E, (uint64_t)N, kb,
                                                    (uint32_t)QROWS, 1);
  if (!wok) return cudaErrorNotSupported;
  for (int i = 0; i < NXBOX; ++i)
    if (!make_tma_map_u8(&maps.x[i], A, (uint64_t)M, kb, 64u >> i) ||
        !make_tma_map_scales(&maps.sx[i], sfa, (uint64_t)M, sc, 64u >> i))
      return cudaErrorNotSupported;
  QParams p;
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
  p.NB = silu ? p.I / 64 : N / BM;  // 128-row tiles of the arranged scales
  p.NBG = p.NB / 2;                 // 256-row tiles of this kernel
  p.KB = Kd / 256;
  p.early_table = early_table ? 1 : 0;
  p.stall_stage = stall_stage;
  // four stages when they fit with the tile table (E up to ~470), else three
  if (q_smem_bytes<4>(E) <= QSMEM_MAX)
    return silu ? launch_q<true, 4>(maps, p, M, E, st, pdl)
                : launch_q<false, 4>(maps, p, M, E, st, pdl);
  return silu ? launch_q<true, 3>(maps, p, M, E, st, pdl) : launch_q<false, 3>(maps, p, M, E, st, pdl);
}

}  // namespace moe
