// moe_grouped_gemm_block: the grouped FP8 GEMM with block scales — one fp32
// scale per 128 x 128 weight block and one per token per 128 input channels
// (the group_k / group_n path that "Fix one bug in the grouped-gemm triton
// kernel", sglang #6772, Highlights, contrasts with the per-token one):
//   C[r,n] = sum_kb (sum_{k in kb} A[r,k] W[e,n,k]) * sa[r,kb] * sb[e,n/128,kb]
//
// The scales change every 128 channels of K, so the tensor cores cannot keep
// one accumulator across K. A K block is exactly one pipeline stage: the MMA
// thread writes each block's partial sum afresh into one of the TMEM partial
// buffers (2 of 256 columns, or 4 of 128), and the epilogue warps fold it
// into fp32 registers while the MMA fills the next one.
//
// Orientation: tokens are the MMA's M side (128 rows per tile) and weights
// its N side: 256 rows (two weight scale blocks; SiLU: four groups of 32 gate
// rows and the matching 32 up rows = 128 j's, whose gate rows lie in one
// scale block and up rows in another), or 128 when N % 256 != 0. A TMEM lane is
// then one token row, and a K block's factor sa[token,kb] * sb[kb] is one
// scalar per thread (two for SiLU: gate and up), so the fold is plain packed
// FMAs with no per-column factor traffic. Tiles are (expert, weight block,
// chunk of at most 128 of the expert's tokens), the MMA is always M = 128:
// rows past the chunk are computed and dropped.
//
// One persistent CTA per SM (tcgen05.mma.cta_group::1), 384 threads:
//   warp 0      TMA producer (one K block of tokens and weights per stage)
//   warp 1      MMA issuer (K = 32 x 4 per K block) into TMEM partial buffer
//               kb % (512 / weight rows per tile)
//   warps 2, 3  idle (they complete warpgroup 0, which hands its registers
//               to the epilogue)
//   warps 4..11 epilogue: warp w reads TMEM lane quadrant w % 4 (32 token
//               rows) and the columns of its half (w - 4) / 4 (one scale
//               block), folds each K block's partial with its row's factor
//               (holding the half's fp32 sums in registers: 128 with
//               256-row tiles), and at the tile's end writes its row segment
//               (SiLU*mul of its gate/up pairs, or bf16 outputs) through a
//               2 KB shared-memory slot, 8 rows x 64 bytes per store.
// Every wait is bounded.
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

constexpr int TM = 128;                  // token rows per tile (MMA M)
constexpr int EW = 8;                    // epilogue warps (warpgroups 1 and 2)
constexpr int BTHREADS = 128 + 32 * EW;  // warpgroup 0: producer, MMA issuer, two idle
constexpr uint32_t TCOLS = 512;          // the partial buffers: all of TMEM
// Registers: the launch gives every thread LAUNCH_REGS (the most that 384
// threads may have); warpgroup 0 gives back all but WG0_REGS, the epilogue
// warpgroups take EPI_REGS. The split adds up to the launch's total exactly.
constexpr int LAUNCH_REGS = 168;
constexpr int WG0_REGS = 88;
constexpr int EPI_REGS = 208;
static_assert(128 * WG0_REGS + 32 * EW * EPI_REGS == BTHREADS * LAUNCH_REGS,
              "register split must add up to the launch's registers");
constexpr int BLK_CW = 16;  // TMEM columns per epilogue load (32 measured slower)

// NW weight rows per tile (MMA N): 256 when N allows (two scale blocks, a
// quarter fewer bytes staged per MMA), else 128. TMEM holds 512 / NW partial
// buffers; the ring as many 16 KB + NW x 128 B stages as fit.
template <int NW>
struct BCfg {
  static constexpr int NPB = 512 / NW;
  static constexpr int STAGES = NW == 256 ? 4 : 6;
  static constexpr int HALF = NW / 2;  // TMEM columns per epilogue warp
};

template <int NW>
struct BSmem {
  static constexpr int STAGES = BCfg<NW>::STAGES;
  static constexpr int NPB = BCfg<NW>::NPB;
  uint8_t x[STAGES][TM * BK];      // tokens (A), one K block per stage
  uint8_t w[STAGES][NW * BK];      // weights (B)
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t pfull[NPB];   // a K block's partial sum is in TMEM buffer b
  uint64_t pempty[NPB];  // every epilogue warp has read it
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int never;
  int thr_sum[32];        // per-warp tile counts of the tile-table scan
  // each epilogue warp's output staging: 32 rows x 64 bytes, the four 16-byte
  // units of row R at positions u ^ ((R >> 1) & 3) (conflict-free both ways)
  uint4 stage_out[EW][32 * 4];
  int tile_start[MAX_E + 1];
  int offs[MAX_E + 1];
};

struct BParams {
  const float* scale_a;  // [M, KB]
  const float* scale_b;  // [E, N/128, KB]
  const int32_t* offsets;
  void* C;
  int* err;
  int M, N, Kd, E, I, NB, KB;
  int stream_weights;
  int early_table;  // build the tile table before waiting for the previous kernel
};

// acc0/1 += v0/1 * f0/1, two lanes of fp32 at once (each rounded as fmaf).
__device__ __forceinline__ void fma2(float& acc0, float& acc1, float v0, float v1, float f0,
                                     float f1) {
  asm("{\n\t.reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\t"
      "mov.b64 {%0, %1}, c;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "f"(v0), "f"(v1), "f"(f0), "f"(f1));
}

template <bool SILU, int NW>
__global__ void __launch_bounds__(BTHREADS, 1)
    grouped_gemm_block_kernel(const __grid_constant__ Maps maps, const BParams p) {
  using S = BSmem<NW>;
  constexpr int BSTAGES = S::STAGES;
  constexpr int NPB = S::NPB;
  constexpr int HALF = BCfg<NW>::HALF;
  constexpr int JT = NW / 2;  // SiLU: j's per tile (gate/up pairs)
  extern __shared__ uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;
  const int KB = p.KB;

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&maps.w);
    for (int i = 0; i < NXBOX; ++i) ptx::prefetch_tensormap(&maps.x[i]);
    for (int s = 0; s < BSTAGES; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < NPB; ++b) {
      ptx::mbar_init(&sm.pfull[b], 1);
      ptx::mbar_init(&sm.pempty[b], EW);
    }
    ptx::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    sm.never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, TCOLS);
    ptx::tmem_relinquish();
  }
  // (inside a chained forward the offsets of the w2 GEMM were written two
  // kernels earlier, so its table is built before the wait)
  if (!p.early_table) chain_entry();
  build_tile_table<TM, BTHREADS>(sm, p.offsets, E, p.M, p.NB, p.err, tid);
  if (p.early_table) chain_entry();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int total = sm.total_tiles;
  const int ncta = gridDim.x;

  // stages the producer armed (and the phase of the latest arming), for the
  // drain after an abort
  uint32_t armed = 0, armed_par = 0;
  if (warp < 4) ptx::setmaxnreg_dec<WG0_REGS>();
  if (warp == 0) {
    // ======================= TMA producer ===================================
    if (lane == 0) {
      // weights evict-first when every block is read once, or when this
      // expert's tokens fit one chunk; tokens evict-last
      const uint64_t pol_w =
          p.stream_weights ? ptx::policy_evict_first() : ptx::policy_evict_normal();
      const uint64_t pol_w1 = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      uint32_t s = 0, ph = 0;
      bool ok = true;
      for (int g = blockIdx.x; ok && g < total; g += ncta) {
        const TileInfo<TM> t = decode_tile<TM>(sm, E, p.NB, g);
        const int rows = (t.ntok + 15) & ~15;
        const uint32_t bytes = (uint32_t)(NW + rows) * BK;
        const uint64_t pw = t.nch == 1 ? pol_w1 : pol_w;
        const int y0 = t.e * p.N + t.nb * NW;  // bf16 epilogue: the tile's first weight row
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(&sm.empty[s], ph ^ 1u, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&sm.full[s], bytes);
          armed |= 1u << s;
          armed_par = (armed_par & ~(1u << s)) | (ph << s);
          if (SILU) {  // per 32 j: the gate rows, then their up rows
#pragma unroll
            for (int gq = 0; gq < JT / 32; ++gq)
              ptx::tma_load_5d(sm.w[s] + gq * 64 * BK, &maps.w, &sm.full[s], 0,
                               t.nb * JT + gq * 32, 0, kb, t.e, pw);
          } else {
            ptx::tma_load_3d(sm.w[s], &maps.w, &sm.full[s], 0, y0, kb, pw);
          }
          int r = 0;
#pragma unroll
          for (int i = 0; i < NXBOX; ++i) {
            const int box = 64 >> i;
            while (rows - r >= box) {
              ptx::tma_load_2d(sm.x[s] + r * BK, &maps.x[i], &sm.full[s], kb * BK, t.tok0 + r,
                               pol_x);
              r += box;
            }
          }
          if (++s == BSTAGES) {
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
      uint32_t kbg = 0;  // K blocks issued so far (selects the partial buffer)
      bool ok = true, issued = false;
      const uint32_t idesc = ptx::idesc_e4m3_f32(TM, NW);
      for (int g = blockIdx.x; ok && g < total; g += ncta) {
        for (int kb = 0; kb < KB; ++kb, ++kbg) {
          const uint32_t b = kbg % NPB;
          if (!ptx::mbar_wait(&sm.pempty[b], ((kbg / NPB) & 1u) ^ 1u, &sm.abort, WAIT_NS) ||
              !ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem + b * NW;
          const uint32_t a0 = ptx::smem_u32(sm.x[s]);
          const uint32_t b0 = ptx::smem_u32(sm.w[s]);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            ptx::mma_e4m3(d, ptx::sdesc_sw128(a0 + kk * 32), ptx::sdesc_sw128(b0 + kk * 32),
                          idesc, kk != 0 ? 1u : 0u);
          issued = true;
          ptx::mma_commit(&sm.empty[s]);
          ptx::mma_commit(&sm.pfull[b]);
          if (++s == BSTAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
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
  } else if (warp >= 4) {
    // ======================= epilogue (warps 4..11) =========================
    // (the increase sits inside the branch, so the compiler sees that only
    // the epilogue code runs with the larger register budget)
    ptx::setmaxnreg_inc<EPI_REGS>();
    const int q = warp & 3;              // TMEM lane quadrant: token rows 32q .. 32q+31
    const int ch = (warp - 4) >> 2;      // column half: TMEM columns HALF*ch ..
    const int r = q * 32 + lane;         // this thread's token row in the tile
    const int NBk = p.N / BM;            // weight scale blocks along N
    // TMEM is read in chunks of CW columns, one chunk in flight while the
    // previous one is folded; SiLU: columns 64g .. 64g+31 gate, 64g+32 .. up
    constexpr int CW = BLK_CW;
    constexpr int NC = HALF / CW;
    uint32_t kbg = 0;
    bool stop = false;
    uint32_t va[CW], vb[CW];  // TMEM chunk registers (vb's first contents are never used)
#pragma unroll
    for (int i = 0; i < CW; ++i) vb[i] = 0u;
    for (int g = blockIdx.x; !stop && g < total; g += ncta) {
      const TileInfo<TM> t = decode_tile<TM>(sm, E, p.NB, g);
      const bool valid = r < t.ntok;
      const float* sa = p.scale_a + (int64_t)(t.tok0 + (valid ? r : 0)) * KB;
      // the weight scale blocks of this half's columns: one 128-row block
      // (bf16 out), or the block of its gate rows and of its up rows (SiLU:
      // the half holds j0 + HALF/2*ch .. for both)
      const float* sbe = p.scale_b + (int64_t)t.e * NBk * KB;
      const int jh = t.nb * JT + ch * (HALF / 2);  // SiLU: first j of the half
      const float* sbg = sbe + (SILU ? jh / BM : (t.nb * NW + ch * HALF) / BM) * KB;
      const float* sbu = sbe + (SILU ? (p.I + jh) / BM : (t.nb * NW + ch * HALF) / BM) * KB;
      float acc[HALF];
#pragma unroll
      for (int i = 0; i < HALF; ++i) acc[i] = 0.0f;
      // the scales of the next K block, loaded one block ahead
      float na = valid ? __ldg(sa) : 0.0f;
      float ng = __ldg(sbg);
      float nu = SILU ? __ldg(sbu) : 0.0f;
      for (int kb = 0; kb < KB; ++kb, ++kbg) {
        const uint32_t b = kbg % NPB;
        const float fg = na * ng;
        const float fu = SILU ? na * nu : fg;
        if (kb + 1 < KB) {
          if (valid) na = __ldg(sa + kb + 1);
          ng = __ldg(sbg + kb + 1);
          if (SILU) nu = __ldg(sbu + kb + 1);
        }
        if (!__all_sync(kFull, ptx::mbar_wait(&sm.pfull[b], (kbg / NPB) & 1u, &sm.abort,
                                              WAIT_NS))) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + b * NW + ch * HALF;
        // chunk c + 1 is read from TMEM while chunk c is folded (load, fold
        // and wait in one asm statement)
        ptx::tmem_ld_sync(tb, va);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          uint32_t(&cur)[CW] = (c & 1) ? vb : va;
          uint32_t(&nxt)[CW] = (c & 1) ? va : vb;
          const float f = (SILU && ((c * CW) & 32)) ? fu : fg;
          float(&a)[CW] = *reinterpret_cast<float(*)[CW]>(acc + c * CW);
          if (c + 1 < NC) {
            ptx::tmem_ld_fold(tb + (c + 1) * CW, nxt, cur, a, f);
          } else {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.pempty[b]);  // the buffer is read
#pragma unroll
            for (int i = 0; i < CW; i += 2)
              fma2(a[i], a[i + 1], __uint_as_float(cur[i]), __uint_as_float(cur[i + 1]), f, f);
          }
        }
      }
      if (stop) break;
      // ---- the warp's rows of the tile's output ----
      // Each round stages 64 bytes of each of the warp's 32 rows in shared
      // memory and stores them as 8 rows x 64 contiguous bytes per
      // instruction (a row-per-thread store would touch 32 lines at once).
      const int nrow = min(32, t.ntok - q * 32);  // the warp's valid rows
      if (nrow <= 0) continue;
      const int64_t row0 = t.tok0 + q * 32;
      uint4* st = sm.stage_out[warp - 4];
      auto stage_row = [&](int u, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
        st[lane * 4 + (u ^ ((lane >> 1) & 3))] = make_uint4(w0, w1, w2, w3);
      };
      // the staged 32 x 64 bytes go to rows row0.. of the output, from column col
      auto flush = [&](int64_t ld, int64_t col) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int R = 8 * i + (lane >> 2), U = lane & 3;
          const uint4 v = st[R * 4 + (U ^ ((R >> 1) & 3))];
          if (R < nrow)
            *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.C) + (row0 + R) * ld +
                                      col + U * 8) = v;
        }
        __syncwarp();
      };
      if (SILU) {
        // group gq: gate of j = jh + 32gq + i in columns 64gq + i, its up in
        // 64gq + 32 + i
#pragma unroll
        for (int gq = 0; gq < HALF / 64; ++gq) {
          uint32_t hv[16];
          const float* a = acc + gq * 64;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float g0 = a[i], g1 = a[i + 1];
            hv[i / 2] = pack_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * a[32 + i],
                                    __fdividef(g1, 1.0f + __expf(-g1)) * a[33 + i]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            stage_row(u, hv[4 * u], hv[4 * u + 1], hv[4 * u + 2], hv[4 * u + 3]);
          flush(p.I, jh + gq * 32);
        }
      } else {
#pragma unroll
        for (int k = 0; k < HALF / 32; ++k) {
          const float* a = acc + k * 32;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            stage_row(u, pack_bf16x2(a[8 * u], a[8 * u + 1]), pack_bf16x2(a[8 * u + 2], a[8 * u + 3]),
                      pack_bf16x2(a[8 * u + 4], a[8 * u + 5]),
                      pack_bf16x2(a[8 * u + 6], a[8 * u + 7]));
          flush(p.N, (int64_t)t.nb * NW + ch * HALF + k * 32);
        }
      }
    }
    if (stop) {
      sm.abort = 1;
      flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before();
  __syncthreads();
  // after an abort (whichever role gave up, possibly after the producer had
  // finished its loop), every copy the producer issued lands before the CTA
  // frees its tensor memory and leaves
  if (warp == 0 && lane == 0 && *reinterpret_cast<volatile int*>(&sm.abort))
    for (int i = 0; i < BSTAGES; ++i)
      if ((armed >> i) & 1u)
        ptx::mbar_wait(&sm.full[i], (armed_par >> i) & 1u, &sm.never, DRAIN_NS);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TCOLS);
  }
}

template <bool SILU, int NW>
cudaError_t launch_block_cfg(const Maps& maps, const BParams& p, int M, int E, cudaStream_t st,
                             bool pdl) {
  constexpr size_t smem = sizeof(BSmem<NW>) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = grouped_gemm_block_kernel<SILU, NW>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 64 || !attr_set[dev]) {
      // the warpgroups' register split assumes the launch gives every thread
      // LAUNCH_REGS registers; with fewer the epilogue's increase would wait
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != LAUNCH_REGS) return cudaErrorNotSupported;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (dev < 64) attr_set[dev] = true;
    }
  }
  const long long upper = ((long long)(M + TM - 1) / TM + E) * p.NB;
  const int grid = (int)std::max<long long>(1, std::min<long long>(sm_count(), upper));
  return launch_kernel(kern, dim3(grid), dim3(BTHREADS), smem, st, pdl, maps, p);
}

}  // namespace

cudaError_t launch_grouped_gemm_block(const void* A, const float* scale_a, const void* B,
                                      const float* scale_b, const int32_t* offsets, int M, int N,
                                      int Kd, int E, int epilogue, void* C, int* err,
                                      cudaStream_t st, bool pdl, bool early_table) {
  if (M == 0) return cudaSuccess;
  const bool silu = (epilogue == MOE_EPI_SILU_MUL);
  const bool small = (int64_t)M <= (int64_t)32 * E;  // few rows per expert (decode)
  // one K block per stage (Kd % 128 == 0, checked at the entry point); SiLU:
  // boxes of 32 gate rows and the matching 32 up rows; bf16: the tile's rows
  // in one box
  Maps maps;
  const bool wok =
      silu ? make_tma_map_weights_pairs32(&maps.w, B, (uint64_t)E, (uint64_t)N, (uint64_t)Kd)
           : make_tma_map_weights_rows(&maps.w, B, (uint64_t)E, (uint64_t)N, (uint64_t)Kd,
                                       N % 256 == 0 ? 256u : 128u);
  if (!weights_stage_box((uint64_t)Kd) || !wok) return cudaErrorNotSupported;
  for (int i = 0; i < NXBOX; ++i)
    if (!make_tma_map_u8(&maps.x[i], A, (uint64_t)M, (uint64_t)Kd, 64u >> i))
      return cudaErrorNotSupported;
  BParams p;
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
  // 256 weight rows per tile when N allows it (SiLU: 128 j's, I % 128 == 0
  // always holds here; bf16: N % 256 == 0)
  const bool wide = silu || N % 256 == 0;
  p.NB = silu ? p.I / (wide ? 128 : 64) : N / (wide ? 256 : BM);
  p.KB = Kd / BK;
  p.stream_weights = small ? 1 : 0;
  p.early_table = early_table ? 1 : 0;
  if (wide)
    return silu ? launch_block_cfg<true, 256>(maps, p, M, E, st, pdl)
                : launch_block_cfg<false, 256>(maps, p, M, E, st, pdl);
  return launch_block_cfg<false, 128>(maps, p, M, E, st, pdl);
}

}  // namespace moe
