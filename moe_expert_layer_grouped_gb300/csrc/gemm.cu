// moe_grouped_gemm: FP8 (e4m3) grouped GEMM over expert row segments on the
// 5th-generation tensor cores, with the per-row x per-channel dequantisation
// fused into the epilogue ("Fix one bug in the grouped-gemm triton kernel",
// sglang #6772, Highlights: scale_a is indexed by the row, m_range_start +
// offs_am; "Support token-level quantization for EP MoE", sglang #6782,
// Changelog: per-token scale_a in the grouped GEMM).
//
// Orientation: the weights are the MMA's M side and the tokens its N side
// (D^T = W * A^T). A tile is 128 weight rows x N tokens of one expert, with
// N the expert's remaining tokens rounded up to 16 (at most BNMAX), so an
// expert's token count is padded to a multiple of 16 rather than of 128.
//
// Design (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0      TMA producer: per stage KC chunks of 128 B of K: the tile's
//               128 weight rows of all KC chunks in one box (one box per chunk
//               when Kd % 128 != 0; for SiLU 64 gate rows then the matching
//               64 up rows), and per chunk the tile's tokens (rounded up to
//               16, covered exactly by boxes of 64/32/16 rows),
//               into a STAGES-deep ring, 128-byte swizzled; weight blocks read
//               by one tile only are loaded evict-first, tokens evict-last.
//   warp 1      MMA issuer: tcgen05.mma.cta_group::1.kind::f8f6f4,
//               M=128 x N x K=32, fp32 accumulator in tensor memory; two
//               accumulators (2 x 256 columns) so the epilogue of tile i
//               overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: tcgen05.ld (one weight row per thread, 32 tokens
//               per load), dequantise by scale_a[token] * scale_b[e, row],
//               then bf16 out, or SiLU(gate) * up; the bf16 block is
//               transposed through shared memory so each token row is stored
//               with 16-byte vectors.
// SiLU*mul: a w13 tile holds gate rows [j0, j0+64) in TMEM lanes 0..63 and
// the matching up rows [I+j0, I+j0+64) in lanes 64..127. The warp holding
// gate lanes and the warp holding the same j's up lanes trade alternate
// 32-token chunks through shared memory, so each computes silu(g)*u for half
// of the tokens.
// Tiles are (expert, weight block, token chunk) with the token chunk fastest,
// so the chunks of one expert stream the same weight block at the same time
// and share it through L2. The tile table is derived on the device from the
// expert offsets (no host synchronisation); tokens past the expert's segment
// are never stored.
// Large batches run on CTA pairs (cluster of 2, tcgen05.mma.cta_group::2:
// 256 weight rows x up to 256 tokens, each CTA holding its own weight rows
// and half of the tokens); few tokens per expert use single CTAs with
// 64-token tiles (see launch_grouped_gemm).
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

constexpr int THREADS = 192;
constexpr uint32_t ACC_COLS = 256;  // TMEM columns per accumulator
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
#ifndef PAIR_KC
#define PAIR_KC 2
#define PAIR_STAGES 3
#endif

template <int XROWS, int STAGES, bool SILU, int KC>
struct Smem {
  uint8_t w[STAGES][KC][W_BYTES];     // weights: KC K-chunks of 128 B per stage
  uint8_t x[STAGES][KC][XROWS * BK];  // this CTA's token rows
  float xchg[SILU ? 2 : 1][2][32 * 32];  // SiLU pairs: 2 slots of 32 tokens x 32 lanes
  uint16_t stage_out[4][32 * 32];        // per epilogue warp: bf16 [token][32 columns]
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int never;  // stays 0: abort flag for the drain waits
  int thr_sum[THREADS];
  int tile_start[MAX_E + 1];
  int offs[MAX_E + 1];
};


struct Params {
  const float* scale_a;
  const float* scale_b;
  const int32_t* offsets;
  void* C;
  float* row_amax;
  int* err;
  int M, N, Kd, E, I, NB, KB;
  int stream_weights;  // 1: each weight block is read by one tile (evict-first)
  int stall_stage;     // failure test: CTA 0 never loads its stage with this index (-1: none)
  int w_stage_box;     // the weight map holds a stage per box (else a K chunk)
  int early_table;     // build the tile table before waiting for the previous kernel
  // token rows gathered from a token-order A ([T, Kd], maps.xg): permuted row
  // r is row row_token[r] of it (null: A is in permuted order, maps.x)
  const int32_t* row_token;
  int T;
};

// CS = 1: one CTA per tile of 128 weight rows x N tokens.
// CS = 2: a CTA pair (cluster of 2) computes 256 weight rows x N tokens with
// the 2-SM MMA (tcgen05.mma.cta_group::2, issued by the even CTA): each CTA
// holds its own 128 weight rows (its own weight block) and half of the N
// token rows, and receives its 128 x N slice of the accumulator in its own
// tensor memory, so a CTA moves and stores two thirds of the bytes a single
// CTA would for the same MMA work. Epilogues are per CTA as in CS = 1.
template <int BNMAX, int STAGES, bool SILU, int CS, int KC>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ Maps maps, const Params p) {
  static_assert(CS == 1 || CS == 2, "single CTA or CTA pair");
  constexpr bool PAIR = (CS == 2);
  using S = Smem<BNMAX / CS, STAGES, SILU, KC>;
  const int KS = (p.KB + KC - 1) / KC;  // pipeline stages per tile
  extern __shared__ uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;

  const bool gather = p.row_token != nullptr;
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&maps.w);
    if (gather)
      ptx::prefetch_tensormap(&maps.xg);
    else
      for (int i = 0; i < NXBOX; ++i) ptx::prefetch_tensormap(&maps.x[i]);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sm.full[s], 1);   // pair: only the even CTA's is used
      ptx::mbar_init(&sm.empty[s], 1);  // one (multicast) MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sm.tfull[b], 1);
      ptx::mbar_init(&sm.tempty[b], 128 * CS);  // pair: both CTAs' epilogues
    }
    ptx::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    sm.never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      ptx::tmem_alloc_pair(&sm.tmem_base, TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&sm.tmem_base, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
  const int cluster = blockIdx.x / CS;
  const int nclusters = gridDim.x / CS;
  const int NBG = p.NB / CS;  // weight-block groups per expert
  constexpr uint16_t kPair = 0x3;
  if (PAIR) ptx::cluster_sync();  // the peer's barriers exist before any signal

  // ---- tile table from the expert offsets --------------------------------
  // (inside a chained forward the offsets of the w2 GEMM were written two
  // kernels earlier, so its table is built before the wait)
  if (!p.early_table) chain_entry();
  build_tile_table<BNMAX, THREADS>(sm, p.offsets, E, p.M, NBG, p.err, tid);
  if (p.early_table) chain_entry();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int total = sm.total_tiles;  // after the barrier above

  // stages the producer armed (and the phase of the latest arming), for the
  // drain after an abort
  uint32_t armed = 0, armed_par = 0;
  if (warp == 0) {
    // ======================= TMA producer ===================================
    // lane 0 waits for free stages, arms them and loads the weights (and the
    // token boxes); with a token-order A every lane gathers four token rows
    // of the stage per instruction (G4 groups of four rows per lane)
    constexpr int G4 = (BNMAX / CS + 127) / 128;
    // weights: evict-first when a block is read once (every block when
    // streaming; otherwise the blocks of experts whose tokens fit one
    // chunk), so they do not push the token tiles, read once per weight
    // block group, out of L2
    const uint64_t pol_w = p.stream_weights ? ptx::policy_evict_first() : ptx::policy_evict_normal();
    const uint64_t pol_w1 = ptx::policy_evict_first();
    const uint64_t pol_x = ptx::policy_evict_last();
    uint32_t s = 0, ph = 0;
    int gstage = 0;  // stages issued by this CTA
    bool ok = true;
    for (int g = cluster; ok && g < total; g += nclusters) {
      const TileInfo<BNMAX> t = decode_tile<BNMAX>(sm, E, NBG, g);
      const int nb = t.nb * CS + rank;
      // token rows of the MMA (N): a multiple of 16, of 32 for a pair so
      // each CTA holds N/2 rows; this CTA loads rows [rank*half, +half)
      const int rows = PAIR ? (t.ntok + 31) & ~31 : (t.ntok + 15) & ~15;
      const int half = rows / CS;
      const uint32_t bytes = KC * (CS * W_BYTES + (uint32_t)rows * BK);  // all CTAs' loads
      const int y0 = t.e * p.N + nb * BM;  // bf16 epilogue: the tile's first weight row
      // gather: this lane's token rows (rows past the tile: row T, outside
      // the tensor, read as zeros)
      int tr[G4][4];
      if (gather) {
#pragma unroll
        for (int q = 0; q < G4; ++q)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = (q * 32 + lane) * 4 + i;  // row within this CTA's half
            const int rt = rank * half + rr;         // row within the tile
            tr[q][i] = (rr < half && rt < t.ntok) ? __ldg(p.row_token + t.tok0 + rt) : p.T;
          }
      }
      for (int ks = 0; ks < KS; ++ks) {
        // every lane waits (each then sees the stage free before it issues)
        const bool got = ptx::mbar_wait(&sm.empty[s], ph ^ 1u, &sm.abort, WAIT_NS);
        if (!__all_sync(kFull, got)) {
          ok = false;
          break;
        }
        // pair: completions count on the even CTA's barrier
        const uint32_t fb = PAIR ? ptx::map_to_rank(ptx::smem_u32(&sm.full[s]), 0) : 0u;
        // failure test: the stage is armed but its bytes never come, so the
        // bounded waits run out
        const bool stall = blockIdx.x == 0 && gstage++ == p.stall_stage;
        if (lane == 0) {
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(&sm.full[s], bytes);
            armed |= 1u << s;
            armed_par = (armed_par & ~(1u << s)) | (ph << s);
          }
          if (!stall && p.w_stage_box) {  // the stage's KC weight chunks in one box
            const uint64_t pw = t.nch == 1 ? pol_w1 : pol_w;
            if (PAIR) {
              if (SILU)  // per chunk 64 gate rows, then the matching 64 up rows
                ptx::tma_load_5d_pair(sm.w[s][0], &maps.w, fb, 0, nb * 64, 0, ks * KC, t.e, pw);
              else  // per chunk the tile's 128 contiguous weight rows
                ptx::tma_load_3d_pair(sm.w[s][0], &maps.w, fb, 0, y0, ks * KC, pw);
            } else {
              if (SILU)
                ptx::tma_load_5d(sm.w[s][0], &maps.w, &sm.full[s], 0, nb * 64, 0, ks * KC, t.e, pw);
              else
                ptx::tma_load_3d(sm.w[s][0], &maps.w, &sm.full[s], 0, y0, ks * KC, pw);
            }
          }
#pragma unroll
          for (int kc = 0; kc < (stall ? 0 : KC); ++kc) {
            const int kx = (ks * KC + kc) * BK;  // past Kd: zero-filled, adds nothing
            uint8_t* xdst = sm.x[s][kc];
            if (!p.w_stage_box) {  // Kd % 128 != 0: the chunk's weights on their own
              const uint64_t pw = t.nch == 1 ? pol_w1 : pol_w;
              if (PAIR) {
                if (SILU)
                  ptx::tma_load_4d_pair(sm.w[s][kc], &maps.w, fb, kx, nb * 64, 0, t.e, pw);
                else
                  ptx::tma_load_2d_pair(sm.w[s][kc], &maps.w, fb, kx, y0, pw);
              } else {
                if (SILU)
                  ptx::tma_load_4d(sm.w[s][kc], &maps.w, &sm.full[s], kx, nb * 64, 0, t.e, pw);
                else
                  ptx::tma_load_2d(sm.w[s][kc], &maps.w, &sm.full[s], kx, y0, pw);
              }
            }
            if (gather) continue;
            if (PAIR) {
              int r = 0;
#pragma unroll
              for (int i = 0; i < NXBOX; ++i) {
                const int box = 64 >> i;
                while (half - r >= box) {
                  ptx::tma_load_2d_pair(xdst + r * BK, &maps.x[i], fb, kx,
                                        t.tok0 + rank * half + r, pol_x);
                  r += box;
                }
              }
            } else {
              int r = 0;
#pragma unroll
              for (int i = 0; i < NXBOX; ++i) {
                const int box = 64 >> i;
                while (rows - r >= box) {
                  ptx::tma_load_2d(xdst + r * BK, &maps.x[i], &sm.full[s], kx, t.tok0 + r, pol_x);
                  r += box;
                }
              }
            }
          }
        }
        if (gather && !stall) {
#pragma unroll
          for (int kc = 0; kc < KC; ++kc) {
            const int kx = (ks * KC + kc) * BK;
#pragma unroll
            for (int q = 0; q < G4; ++q) {
              const int rr = (q * 32 + lane) * 4;
              if (rr < half) {
                uint8_t* xdst = sm.x[s][kc] + rr * BK;
                if (PAIR)
                  ptx::tma_gather4_pair(xdst, &maps.xg, fb, kx, tr[q][0], tr[q][1], tr[q][2],
                                        tr[q][3], pol_x);
                else
                  ptx::tma_gather4(xdst, &maps.xg, &sm.full[s], kx, tr[q][0], tr[q][1],
                                   tr[q][2], tr[q][3], pol_x);
              }
            }
          }
        }
        if (++s == STAGES) {
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
    if (lane == 0 && rank == 0) {  // pair: the even CTA issues for both
      uint32_t s = 0, ph = 0;
      bool ok = true, issued = false;
      int iter = 0;
      for (int g = cluster; ok && g < total; g += nclusters, ++iter) {
        const TileInfo<BNMAX> t = decode_tile<BNMAX>(sm, E, NBG, g);
        const int n_mma = PAIR ? (t.ntok + 31) & ~31 : (t.ntok + 15) & ~15;
        const uint32_t idesc = ptx::idesc_e4m3_f32(BM * CS, n_mma);
        const int b = iter & 1;
        const uint32_t tph = (iter >> 1) & 1;
        if (!ptx::mbar_wait(&sm.tempty[b], tph ^ 1u, &sm.abort, WAIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)b * ACC_COLS;
        for (int ks = 0; ks < KS; ++ks) {
          if (!ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int kc = 0; kc < KC; ++kc) {
            const uint32_t a0 = ptx::smem_u32(sm.w[s][kc]);
            const uint32_t b0 = ptx::smem_u32(sm.x[s][kc]);
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk) {
              const uint32_t acc = (ks | kc | kk) != 0 ? 1u : 0u;
              if (PAIR)
                ptx::mma_e4m3_pair(d, ptx::sdesc_sw128(a0 + kk * 32),
                                   ptx::sdesc_sw128(b0 + kk * 32), idesc, acc);
              else
                ptx::mma_e4m3(d, ptx::sdesc_sw128(a0 + kk * 32), ptx::sdesc_sw128(b0 + kk * 32),
                              idesc, acc);
            }
          }
          issued = true;
          if (PAIR)
            ptx::mma_commit_pair_mcast(&sm.empty[s], kPair);  // frees the stage in both CTAs
          else
            ptx::mma_commit(&sm.empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR)
          ptx::mma_commit_pair_mcast(&sm.tfull[b], kPair);  // both CTAs' epilogues
        else
          ptx::mma_commit(&sm.tfull[b]);
      }
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        if (issued) {
          if (PAIR)
            ptx::mma_commit_pair_mcast(&sm.drain, 0x1);
          else
            ptx::mma_commit(&sm.drain);
          ptx::mbar_wait(&sm.drain, 0, &sm.never, DRAIN_NS);
        }
      }
    }
  } else {
    // ======================= epilogue (warps 2..5) ==========================
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int iter = 0;
    for (int g = cluster; g < total; g += nclusters, ++iter) {
      TileInfo<BNMAX> t = decode_tile<BNMAX>(sm, E, NBG, g);
      t.nb = t.nb * CS + rank;
      const int b = iter & 1;
      const uint32_t tph = (iter >> 1) & 1;
      bool ok = ptx::mbar_wait(&sm.tfull[b], tph, &sm.abort, WAIT_NS);
      ok = __all_sync(kFull, ok);
      // the two warps of a SiLU exchange pair leave together or not at all
      if (SILU) ok = !bar_red_or(1 + (q & 1), 64, !ok);
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * ACC_COLS;
      const int nchunk = (t.ntok + 31) >> 5;
      const int64_t e = t.e;
      if (SILU) {
        const int I = p.I;
        const int pair = q & 1;           // which 32 of the tile's 64 j
        const bool holds_gate = q < 2;    // lanes 0..63 gate, 64..127 up
        const int j = t.nb * 64 + pair * 32 + lane;
        const bool jv = j < I;
        const float sg = jv ? __ldg(p.scale_b + e * p.N + j) : 0.0f;
        const float su = jv ? __ldg(p.scale_b + e * p.N + I + j) : 0.0f;
        __nv_bfloat16* hbase = reinterpret_cast<__nv_bfloat16*>(p.C);
        // of every 32-token chunk the gate holder computes tokens 0..15 and
        // the up holder tokens 16..31; each hands the other its half
        const int mine0 = holds_gate ? 0 : 16;
        uint16_t* ost = sm.stage_out[q];
        const int jrow = t.nb * 64 + pair * 32;  // first j of this warp's 32
        const bool amax = p.row_amax != nullptr;
        // the next chunk's TMEM load is in flight while this one is processed
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tbase, v);
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          ptx::tmem_ld_wait();
          ptx::reg_fence(v);
          float* give = sm.xchg[pair][c & 1] + (holds_gate ? 16 * 32 : 0);
          const float* take = sm.xchg[pair][c & 1] + (holds_gate ? 0 : 16 * 32);
          float own_v[16];  // this warp's half of the chunk, the other half goes out
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float lo = __uint_as_float(v[i]), hi = __uint_as_float(v[16 + i]);
            own_v[i] = holds_gate ? lo : hi;
            give[i * 32 + lane] = holds_gate ? hi : lo;
          }
          if (c + 1 < nchunk) ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * 32, v);
          bar_sync_named(1 + pair, 64);
          const int tk0 = c * 32 + mine0;
          const float sa_l =
              (lane < 16 && tk0 + lane < t.ntok) ? __ldg(p.scale_a + t.tok0 + tk0 + lane) : 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float other = take[i * 32 + lane];
            const float sa = __shfl_sync(kFull, sa_l, i);
            const float g = (holds_gate ? own_v[i] : other) * sa * sg;
            const float u = (holds_gate ? other : own_v[i]) * sa * su;
            // silu(g) * u; the result is rounded to bf16, so a fast divide
            // (2 ulp) is well inside its precision
            const __nv_bfloat16 hb = __float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * u);
            ost[i * 32 + lane] = __bfloat16_as_ushort(hb);
            if (amax) {
              const float m = warp_max(jv ? fabsf(__bfloat162float(hb)) : 0.0f);
              if (lane == 0 && tk0 + i < t.ntok)
                atomicMax(reinterpret_cast<int*>(p.row_amax + t.tok0 + tk0 + i),
                          __float_as_int(m));
            }
          }
          __syncwarp();
          // 16 tokens x 32 j: four lanes per token row, 16 bytes each
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
        // the partner must be done reading this tile's slots before the next
        // tile overwrites them
        bar_sync_named(1 + pair, 64);
      } else {
        const int N = p.N;
        const int ncol0 = t.nb * BM + q * 32;  // first column of this warp's 32
        const int n = ncol0 + lane;
        const bool nv = n < N;
        const float sb = nv ? __ldg(p.scale_b + e * N + n) : 0.0f;
        uint16_t* ost = sm.stage_out[q];
        __nv_bfloat16* cbase = reinterpret_cast<__nv_bfloat16*>(p.C);
        // the next chunk's TMEM load is in flight while this one is stored
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
          const float sa_l = (tk0 + lane < t.ntok) ? __ldg(p.scale_a + t.tok0 + tk0 + lane) : 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float sa = __shfl_sync(kFull, sa_l, i);
            ost[i * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(f[i] * sa * sb));
          }
          __syncwarp();
          // 32 tokens x 32 columns: four lanes per token row, 16 bytes each
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
      if (PAIR && rank != 0)
        ptx::mbar_arrive_cluster(ptx::map_to_rank(ptx::smem_u32(&sm.tempty[b]), 0));
      else
        ptx::mbar_arrive(&sm.tempty[b]);
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before();
  __syncthreads();
  // after an abort (whichever role gave up, possibly after the producer had
  // finished its loop), every copy the producer issued lands before the CTA
  // frees its tensor memory and leaves
  if (warp == 0 && lane == 0 && *reinterpret_cast<volatile int*>(&sm.abort))
    for (int i = 0; i < STAGES; ++i)
      if ((armed >> i) & 1u)
        ptx::mbar_wait(&sm.full[i], (armed_par >> i) & 1u, &sm.never, DRAIN_NS);
  if (PAIR) {
    // both CTAs are done with the shared accumulator before it is freed, and
    // neither leaves while the other may still signal its barriers
    ptx::cluster_sync();
    if (warp == 1) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
    ptx::cluster_sync();
  } else if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- host side ---------------------------------------------------------------
template <int BNMAX, int STAGES, bool SILU, int CS, int KC>
cudaError_t launch_cfg(const Maps& maps, const Params& p, int M, int E, cudaStream_t st,
                       bool pdl) {
  constexpr size_t smem = sizeof(Smem<BNMAX / CS, STAGES, SILU, KC>) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = grouped_gemm_kernel<BNMAX, STAGES, SILU, CS, KC>;
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
  const long long upper = ((long long)(M + BNMAX - 1) / BNMAX + E) * (p.NB / CS) * CS;
  int grid = (int)std::min<long long>(sm_count(), upper);
  grid = std::max(CS, grid / CS * CS);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (CS > 1) {
    // a persistent grid of pairs must be co-resident: no more clusters than
    // the GPU can hold at once
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) == cudaSuccess && nclusters > 0)
      cfg.gridDim = dim3(std::min(grid, nclusters * CS));
  }
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

}  // namespace

namespace gemm_common {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

namespace {

// Encodes a u8 tensor map (128-byte swizzle, L2 256-byte promotion, zero fill
// outside the tensor). Encoded maps are cached by (address, shape, strides,
// box, device) so repeated calls on the same buffers skip the driver.
bool encode_u8(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
               const cuuint64_t* strides, const cuuint32_t* box,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  struct Entry {
    const void* base;
    int rank, dev, swizzle;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5];
    CUtensorMap map;
  };
  auto same = [&](const Entry& c, int dev) {
    if (c.base != base || c.rank != rank || c.dev != dev || c.swizzle != (int)swizzle)
      return false;
    for (int i = 0; i < rank; ++i)
      if (c.dims[i] != dims[i] || c.box[i] != box[i] || (i + 1 < rank && c.strides[i] != strides[i]))
        return false;
    return true;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& c : cache)
      if (same(c, dev)) {
        *m = c.map;
        return true;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), dims,
         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry e = {};
  e.base = base;
  e.rank = rank;
  e.dev = dev;
  e.swizzle = (int)swizzle;
  for (int i = 0; i < rank; ++i) {
    e.dims[i] = dims[i];
    e.box[i] = box[i];
    if (i + 1 < rank) e.strides[i] = strides[i];
  }
  e.map = *m;
  std::lock_guard<std::mutex> lk(mu);
  cache[next] = e;
  next = (next + 1) % 64;
  return true;
}

}  // namespace

bool make_tma_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {BK, box_rows};
  return encode_u8(m, base, 2, dims, strides, box);
}

bool make_tma_map_scales(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {16, box_rows};
  return encode_u8(m, base, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_tma_map_weight_scales(CUtensorMap* m, const void* base, bool silu, uint64_t E,
                                uint64_t N, uint64_t cols) {
  if (silu) {  // [E][2][I][cols]: 64 gate rows, then the matching 64 up rows
    const uint64_t I = N / 2;
    const cuuint64_t dims[4] = {cols, I, 2, E};
    const cuuint64_t strides[3] = {cols, I * cols, 2 * I * cols};
    const cuuint32_t box[4] = {16, 64, 2, 1};
    return encode_u8(m, base, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  const cuuint64_t dims[2] = {cols, E * N};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {16, BM};
  return encode_u8(m, base, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_tma_map_weights_rows(CUtensorMap* m, const void* base, uint64_t E, uint64_t N,
                               uint64_t Kd, uint32_t rows, uint32_t kc) {
  // [Kd/128][E*N][128]: kc 128-byte K chunks of `rows` consecutive rows per box
  const uint64_t KB = Kd / BK;
  const cuuint64_t dims[3] = {BK, E * N, KB};
  const cuuint64_t strides[2] = {Kd, BK};
  const cuuint32_t box[3] = {BK, rows, kc};
  return encode_u8(m, base, 3, dims, strides, box);
}

bool make_tma_map_weights_gateup(CUtensorMap* m, const void* base, uint64_t E, uint64_t N,
                                 uint64_t Kd, uint32_t jrows, uint32_t kc) {
  // [E][Kd/128][2][I][128] (as the SiLU stage view), boxes of jrows gate rows
  // then the matching jrows up rows, for kc 128-byte chunks
  const uint64_t I = N / 2, KB = Kd / BK;
  const cuuint64_t dims[5] = {BK, I, 2, KB, E};
  const cuuint64_t strides[4] = {Kd, I * Kd, BK, 2 * I * Kd};
  const cuuint32_t box[5] = {BK, jrows, 2, kc, 1};
  return encode_u8(m, base, 5, dims, strides, box);
}

bool make_tma_map_weights_pairs32(CUtensorMap* m, const void* base, uint64_t E, uint64_t N,
                                  uint64_t Kd) {
  return make_tma_map_weights_gateup(m, base, E, N, Kd, 32);
}

bool make_tma_map_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {BK, 1};
  return encode_u8(m, base, 2, dims, strides, box);
}

bool make_tma_map_weights(CUtensorMap* m, const void* base, bool silu, uint64_t E, uint64_t N,
                          uint64_t Kd, uint32_t kc) {
  if (!weights_stage_box(Kd)) {  // one chunk per box, zero past Kd
    if (silu) {
      const uint64_t I = N / 2;
      const cuuint64_t dims[4] = {Kd, I, 2, E};
      const cuuint64_t strides[3] = {Kd, I * Kd, 2 * I * Kd};
      const cuuint32_t box[4] = {BK, 64, 2, 1};
      return encode_u8(m, base, 4, dims, strides, box);
    }
    const cuuint64_t dims[2] = {Kd, E * N};
    const cuuint64_t strides[1] = {Kd};
    const cuuint32_t box[2] = {BK, BM};
    return encode_u8(m, base, 2, dims, strides, box);
  }
  const uint64_t KB = Kd / BK;  // 128-byte chunks of K
  if (silu) {
    const uint64_t I = N / 2;
    const cuuint64_t dims[5] = {BK, I, 2, KB, E};
    const cuuint64_t strides[4] = {Kd, I * Kd, BK, 2 * I * Kd};
    const cuuint32_t box[5] = {BK, 64, 2, kc, 1};
    return encode_u8(m, base, 5, dims, strides, box);
  }
  const cuuint64_t dims[3] = {BK, E * N, KB};
  const cuuint64_t strides[2] = {Kd, BK};
  const cuuint32_t box[3] = {BK, BM, kc};
  return encode_u8(m, base, 3, dims, strides, box);
}

}  // namespace gemm_common

bool gemm_many_rows(int M, int E) { return (int64_t)M > (int64_t)32 * E; }

cudaError_t launch_grouped_gemm(const void* A, const float* scale_a, const void* B,
                                const float* scale_b, const int32_t* offsets, int M, int N,
                                int Kd, int E, int epilogue, void* C, float* row_amax, int* err,
                                cudaStream_t st, int stall_stage, bool pdl, bool early_table,
                                const int32_t* row_token, int T) {
  if (M == 0) return cudaSuccess;
  // long K with many rows per expert: pairs with two accumulators per CTA
  // (gemm_wide.cu), which stage each token row half as often
  if (row_token == nullptr && row_amax == nullptr && gemm_wide_applies(M, N, Kd, E, epilogue))
    return launch_grouped_gemm_wide(A, scale_a, B, scale_b, offsets, M, N, Kd, E, epilogue, C,
                                    err, st, pdl, early_table, stall_stage);
  const bool silu = (epilogue == MOE_EPI_SILU_MUL);
  const bool small = !gemm_many_rows(M, E);  // few rows per expert (decode)
  // K chunks per stage of the configuration launched below (the weight box
  // holds one stage)
  const int nb_blocks = silu ? (N / 2 + 63) / 64 : (N + BM - 1) / BM;
  const uint32_t kc = small ? 2u : (nb_blocks % 2 == 0 ? (uint32_t)PAIR_KC : 1u);
  Maps maps;
  if (!make_tma_map_weights(&maps.w, B, silu, (uint64_t)E, (uint64_t)N, (uint64_t)Kd, kc))
    return cudaErrorNotSupported;
  if (row_token != nullptr) {  // A is [T, Kd] in token order
    if (!make_tma_map_rows(&maps.xg, A, (uint64_t)T, (uint64_t)Kd)) return cudaErrorNotSupported;
  } else {
    for (int i = 0; i < NXBOX; ++i)
      if (!make_tma_map_u8(&maps.x[i], A, (uint64_t)M, (uint64_t)Kd, 64u >> i))
        return cudaErrorNotSupported;
  }
  Params p;
  p.row_token = row_token;
  p.T = T;
  p.scale_a = scale_a;
  p.scale_b = scale_b;
  p.offsets = offsets;
  p.C = C;
  p.row_amax = row_amax;
  p.err = err;
  p.M = M;
  p.N = N;
  p.Kd = Kd;
  p.E = E;
  p.I = N / 2;
  p.NB = silu ? (p.I + 63) / 64 : (N + BM - 1) / BM;
  p.KB = (Kd + BK - 1) / BK;
  p.stream_weights = 0;
  // few rows per expert (decode): small token tiles, weights streamed once
  // through 4 stages of two 128-byte K chunks (256 contiguous bytes of each
  // weight row per stage); many (prefill): tiles of up to 256 tokens
  p.stream_weights = small ? 1 : 0;
  p.stall_stage = stall_stage;
  p.w_stage_box = weights_stage_box((uint64_t)Kd) ? 1 : 0;
  p.early_table = early_table ? 1 : 0;
  if (small)
    return silu ? launch_cfg<64, 4, true, 1, 2>(maps, p, M, E, st, pdl)
                : launch_cfg<64, 4, false, 1, 2>(maps, p, M, E, st, pdl);
  // many tokens per expert: CTA pairs on pairs of weight blocks (2-SM MMA),
  // 3 stages of 2 x (16 KB weights + 16 KB tokens) per CTA
  if (p.NB % 2 == 0)
    return silu ? launch_cfg<256, PAIR_STAGES, true, 2, PAIR_KC>(maps, p, M, E, st, pdl)
                : launch_cfg<256, PAIR_STAGES, false, 2, PAIR_KC>(maps, p, M, E, st, pdl);
  return silu ? launch_cfg<256, 4, true, 1, 1>(maps, p, M, E, st, pdl)
              : launch_cfg<256, 4, false, 1, 1>(maps, p, M, E, st, pdl);
}

}  // namespace moe
