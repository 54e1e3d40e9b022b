// moe_grouped_gemm_block: the grouped FP8 GEMM with block scales — one fp32
// scale per 128 x 128 weight block and one per token per 128 input channels
// (the group_k / group_n path that "Fix one bug in the grouped-gemm triton
// kernel", sglang #6772, Highlights, contrasts with the per-token one):
//   C[r,n] = sum_kb (sum_{k in kb} A[r,k] W[e,n,k]) * sa[r,kb] * sb[e,n/128,kb]
//
// The scales change every 128 channels of K, so the tensor cores cannot keep
// one accumulator across K. A K block is exactly one pipeline stage: the MMA
// thread writes each block's partial sum afresh into one of four TMEM
// buffers, and the epilogue warps fold it into fp32 registers while the MMA
// fills the next buffers.
//
// Orientation: tokens are the MMA's M side (128 rows per tile) and weights
// its N side (128 rows = one weight scale block; SiLU: 32 gate rows, the
// matching 32 up rows, the next 32 gate rows, their 32 up rows = 64 j's whose
// gate rows lie in one scale block and up rows in another). A TMEM lane is
// then one token row, and a K block's factor sa[token,kb] * sb[kb] is one
// scalar per thread (two for SiLU: gate and up), so the fold is plain packed
// FMAs with no per-column factor traffic. Tiles are (expert, weight block,
// chunk of at most 128 of the expert's tokens), the MMA is always M = 128:
// rows past the chunk are computed and dropped.
//
// One persistent CTA per SM (tcgen05.mma.cta_group::1), 320 threads:
//   warp 0      TMA producer (one K block of tokens and weights per stage)
//   warp 1      MMA issuer (K = 32 x 4 per K block) into TMEM buffer kb % 4
//   warps 2..9  epilogue: warp w reads TMEM lane quadrant w % 4 (32 token
//               rows) and the 64 columns of its half (w - 2) / 4, folds each
//               K block's partial with its row's factor, and at the tile's end
//               writes its row segment (SiLU*mul of its 32 gate/up pairs, or
//               64 bf16 outputs) with 16-byte stores.
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
constexpr int EW = 8;                    // epilogue warps
constexpr int BTHREADS = 64 + 32 * EW;   // producer, MMA issuer, epilogue
constexpr int NPB = 4;                   // TMEM partial buffers of BM columns
constexpr uint32_t TCOLS = NPB * BM;     // 512
constexpr int BSTAGES = 6;

struct BSmem {
  uint8_t x[BSTAGES][TM * BK];      // tokens (A), one K block per stage
  uint8_t w[BSTAGES][W_BYTES];      // weights (B)
  uint64_t full[BSTAGES];
  uint64_t empty[BSTAGES];
  uint64_t pfull[NPB];   // a K block's partial sum is in TMEM buffer b
  uint64_t pempty[NPB];  // every epilogue warp has read it
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int never;
  int thr_sum[BTHREADS];
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

template <bool SILU>
__global__ void __launch_bounds__(BTHREADS, 1)
    grouped_gemm_block_kernel(const __grid_constant__ Maps maps, const BParams p) {
  extern __shared__ uint8_t smem_raw[];
  BSmem& sm = *reinterpret_cast<BSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
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
        const uint32_t bytes = W_BYTES + (uint32_t)rows * BK;
        const uint64_t pw = t.nch == 1 ? pol_w1 : pol_w;
        const int y0 = t.e * p.N + t.nb * BM;  // bf16 epilogue: the tile's first weight row
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(&sm.empty[s], ph ^ 1u, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&sm.full[s], bytes);
          armed |= 1u << s;
          armed_par = (armed_par & ~(1u << s)) | (ph << s);
          if (SILU) {  // gate rows j0..j0+31 and their up rows, then j0+32..j0+63
            ptx::tma_load_5d(sm.w[s], &maps.w, &sm.full[s], 0, t.nb * 64, 0, kb, t.e, pw);
            ptx::tma_load_5d(sm.w[s] + 64 * BK, &maps.w, &sm.full[s], 0, t.nb * 64 + 32, 0, kb,
                             t.e, pw);
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
      const uint32_t idesc = ptx::idesc_e4m3_f32(TM, BM);
      for (int g = blockIdx.x; ok && g < total; g += ncta) {
        for (int kb = 0; kb < KB; ++kb, ++kbg) {
          const uint32_t b = kbg % NPB;
          if (!ptx::mbar_wait(&sm.pempty[b], ((kbg / NPB) & 1u) ^ 1u, &sm.abort, WAIT_NS) ||
              !ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem + b * BM;
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
  } else {
    // ======================= epilogue (warps 2..9) ==========================
    const int q = warp & 3;              // TMEM lane quadrant: token rows 32q .. 32q+31
    const int ch = (warp - 2) >> 2;      // column half: TMEM columns 64ch .. 64ch+63
    const int r = q * 32 + lane;         // this thread's token row in the tile
    const int NBk = p.N / BM;            // weight scale blocks along N
    uint32_t kbg = 0;
    bool stop = false;
    for (int g = blockIdx.x; !stop && g < total; g += ncta) {
      const TileInfo<TM> t = decode_tile<TM>(sm, E, p.NB, g);
      const bool valid = r < t.ntok;
      const float* sa = p.scale_a + (int64_t)(t.tok0 + (valid ? r : 0)) * KB;
      // the weight scale blocks of the tile's columns: the 128-row block
      // (bf16 out), or the gate rows' block and the up rows' block (SiLU)
      const float* sbe = p.scale_b + (int64_t)t.e * NBk * KB;
      const float* sbg = sbe + (SILU ? (t.nb * 64) / BM : t.nb) * KB;
      const float* sbu = sbe + (SILU ? (p.I + t.nb * 64) / BM : t.nb) * KB;
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
      float fa = valid ? __ldg(sa) : 0.0f;  // this row's scale of the next K block
      for (int kb = 0; kb < KB; ++kb, ++kbg) {
        const uint32_t b = kbg % NPB;
        const float fg = fa * __ldg(sbg + kb);
        const float fu = SILU ? fa * __ldg(sbu + kb) : fg;
        if (kb + 1 < KB && valid) fa = __ldg(sa + kb + 1);
        if (!__all_sync(kFull, ptx::mbar_wait(&sm.pfull[b], (kbg / NPB) & 1u, &sm.abort,
                                              WAIT_NS))) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + b * BM + ch * 64;
        uint32_t v0[32], v1[32];
        ptx::tmem_ld_32x32b_x32(tb, v0);
        ptx::tmem_ld_32x32b_x32(tb + 32, v1);
        ptx::tmem_ld_wait();
        ptx::reg_fence(v0);
        ptx::reg_fence(v1);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.pempty[b]);  // the buffer is read
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          fma2(acc[i], acc[i + 1], __uint_as_float(v0[i]), __uint_as_float(v0[i + 1]), fg, fg);
          fma2(acc[32 + i], acc[33 + i], __uint_as_float(v1[i]), __uint_as_float(v1[i + 1]),
               fu, fu);
        }
      }
      if (stop) break;
      // ---- this thread's row segment of the tile's output ----
      if (!valid) continue;
      const int64_t tok = t.tok0 + r;
      if (SILU) {
        // columns 0..31 of the half: gate of j = j0 + 32ch + i, 32..63: its up
        uint32_t hv[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float g0 = acc[i], g1 = acc[i + 1];
          hv[i / 2] = pack_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * acc[32 + i],
                                  __fdividef(g1, 1.0f + __expf(-g1)) * acc[33 + i]);
        }
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.C) +
                                              tok * p.I + t.nb * 64 + ch * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_uint4(hv[4 * k], hv[4 * k + 1], hv[4 * k + 2], hv[4 * k + 3]);
      } else {
        uint32_t ov[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) ov[i / 2] = pack_bf16x2(acc[i], acc[i + 1]);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.C) +
                                              tok * p.N + t.nb * BM + ch * 64);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dst[k] = make_uint4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
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

template <bool SILU>
cudaError_t launch_block_cfg(const Maps& maps, const BParams& p, int M, int E, cudaStream_t st,
                             bool pdl) {
  constexpr size_t smem = sizeof(BSmem) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = grouped_gemm_block_kernel<SILU>;
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
  // boxes of 32 gate rows and the matching 32 up rows
  Maps maps;
  const bool wok =
      silu ? make_tma_map_weights_pairs32(&maps.w, B, (uint64_t)E, (uint64_t)N, (uint64_t)Kd)
           : make_tma_map_weights(&maps.w, B, false, (uint64_t)E, (uint64_t)N, (uint64_t)Kd, 1);
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
  p.NB = silu ? p.I / 64 : N / BM;
  p.KB = Kd / BK;
  p.stream_weights = small ? 1 : 0;
  p.early_table = early_table ? 1 : 0;
  return silu ? launch_block_cfg<true>(maps, p, M, E, st, pdl)
              : launch_block_cfg<false>(maps, p, M, E, st, pdl);
}

}  // namespace moe
