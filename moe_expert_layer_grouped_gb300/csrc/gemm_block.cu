// moe_grouped_gemm_block: the grouped FP8 GEMM with block scales — one fp32
// scale per 128 x 128 weight block and one per token per 128 input channels
// (the group_k / group_n path that "Fix one bug in the grouped-gemm triton
// kernel", sglang #6772, Highlights, contrasts with the per-token one):
//   C[r,n] = sum_kb (sum_{k in kb} A[r,k] W[e,n,k]) * sa[r,kb] * sb[e,n/128,kb]
//
// The scales change every 128 channels of K, so the tensor cores cannot keep
// one accumulator across K. A K block is exactly one pipeline stage: the MMA
// thread writes each block's partial sum afresh into one of up to four TMEM
// buffers, and the epilogue warps fold it into fp32 registers with its
// factor sa[token,kb] * sb[kb] while the MMA fills the next buffers.
//
// Orientation and tiles as in moe_grouped_gemm: weights on the MMA's M side
// (128 rows per tile, which is one weight scale block), tokens on N (at most
// BNMAX per tile, 16-token granularity). One persistent CTA per SM
// (tcgen05.mma.cta_group::1), 352 threads:
//   warp 0      TMA producer (one K block of weights and tokens per stage;
//               the weights of a K block in one box, as in moe_grouped_gemm)
//   warp 1      MMA issuer (K=32 x 4 per K block)
//   warps 2..9  epilogue: warp w reads TMEM lane quadrant w % 4 and the
//               32-column token chunks cg, cg + 2, ... (cg = its column
//               group, so ragged tiles split evenly) and accumulates with
//               packed fp32 FMAs; it holds nothing but its accumulators and
//               the TMEM values in flight
//   warp 10     scale warp: per K block, the factor rows
//               sa[token,kb] * sb[kb] of the tile's token columns (SiLU: one
//               for the gate block, one for the up block) into the slot of
//               the partial buffer the block goes to; it reads four K blocks
//               of scales per 16-byte load (each lane's token row is its own
//               cache line), the next four while these are used
// SiLU*mul: gate rows sit in TMEM lanes 0..63 and up rows in 64..127; the two
// warps holding the same j for the same columns trade half of each 32-token
// chunk through shared memory, and each stages its bf16 results in the slot
// it has just read before the 16-byte stores.
// Every wait is bounded; the two warps of a SiLU exchange pair take the abort
// decision together through bar.red so neither is left at a named barrier.
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

constexpr int CG = 2;                    // epilogue column groups
constexpr int EW = 4 * CG;               // epilogue warps
constexpr int BTHREADS = 96 + 32 * EW;   // producer, MMA issuer, epilogue, scale warp
constexpr int SCALE_WARP = 2 + EW;
constexpr int BAR_PAIR = 2;              // named barriers 2..5: the SiLU exchange pairs

// TMEM partial buffers: all 512 columns, at most 4 (the MMA runs up to
// NPB - 1 K blocks ahead of the epilogue).
template <int BNMAX>
__host__ __device__ constexpr int npb() {
  return 512 / BNMAX > 4 ? 4 : 512 / BNMAX;
}

template <int BNMAX, int STAGES, int NF>
struct BSmem {
  uint8_t w[STAGES][W_BYTES];        // weights, one K block per stage
  uint8_t x[STAGES][BNMAX * BK];     // tokens
  // per partial buffer: sa[token,kb] * sb[kb] of the tile's token columns, one
  // row per weight scale block of the tile's rows (SiLU: gate, up)
  float fs[npb<BNMAX>()][NF][BNMAX];
  uint32_t scr[EW][16 * 32];         // per epilogue warp: SiLU exchange / bf16 staging
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t pfull[npb<BNMAX>()];   // a K block's partial sum is in TMEM buffer b
  uint64_t pempty[npb<BNMAX>()];  // every epilogue warp has read it
  uint64_t sfull[npb<BNMAX>()];   // the factor rows of slot b are written
  uint64_t sempty[npb<BNMAX>()];  // every epilogue warp has read them
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

template <int BNMAX, int STAGES, bool SILU>
__global__ void __launch_bounds__(BTHREADS, 1)
    grouped_gemm_block_kernel(const __grid_constant__ Maps maps, const BParams p) {
  constexpr int NF = SILU ? 2 : 1;
  using S = BSmem<BNMAX, STAGES, NF>;
  constexpr int NPB = npb<BNMAX>();
  constexpr uint32_t TCOLS = NPB * BNMAX;  // the partial buffers
  static_assert(TCOLS >= 32 && TCOLS <= 512 && (TCOLS & (TCOLS - 1)) == 0,
                "tensor memory is allocated in powers of two from 32 to 512 columns");
  constexpr int NCH = BNMAX / 32 / CG;  // 32-column chunks per epilogue warp
  constexpr int HC = NCH * 32;          // its token columns
  static_assert(NCH >= 1 && NCH * CG * 32 == BNMAX, "tile shape");
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
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < NPB; ++b) {
      ptx::mbar_init(&sm.pfull[b], 1);
      ptx::mbar_init(&sm.pempty[b], EW);
      ptx::mbar_init(&sm.sfull[b], 1);
      ptx::mbar_init(&sm.sempty[b], EW);
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
  build_tile_table<BNMAX, BTHREADS>(sm, p.offsets, E, p.M, p.NB, p.err, tid);
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
        const TileInfo<BNMAX> t = decode_tile<BNMAX>(sm, E, p.NB, g);
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
          const int kx = kb * BK;
          if (SILU)  // 64 gate rows, then the matching 64 up rows
            ptx::tma_load_5d(sm.w[s], &maps.w, &sm.full[s], 0, t.nb * 64, 0, kb, t.e, pw);
          else
            ptx::tma_load_3d(sm.w[s], &maps.w, &sm.full[s], 0, y0, kb, pw);
          int r = 0;
#pragma unroll
          for (int i = 0; i < NXBOX; ++i) {
            const int box = 64 >> i;
            while (rows - r >= box) {
              ptx::tma_load_2d(sm.x[s] + r * BK, &maps.x[i], &sm.full[s], kx, t.tok0 + r, pol_x);
              r += box;
            }
          }
          if (++s == STAGES) {
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
      for (int g = blockIdx.x; ok && g < total; g += ncta) {
        const TileInfo<BNMAX> t = decode_tile<BNMAX>(sm, E, p.NB, g);
        const uint32_t idesc = ptx::idesc_e4m3_f32(BM, (t.ntok + 15) & ~15);
        for (int kb = 0; kb < KB; ++kb, ++kbg) {
          const uint32_t b = kbg % NPB;
          if (!ptx::mbar_wait(&sm.pempty[b], ((kbg / NPB) & 1u) ^ 1u, &sm.abort, WAIT_NS) ||
              !ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem + b * BNMAX;
          const uint32_t a0 = ptx::smem_u32(sm.w[s]);
          const uint32_t b0 = ptx::smem_u32(sm.x[s]);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            ptx::mma_e4m3(d, ptx::sdesc_sw128(a0 + kk * 32), ptx::sdesc_sw128(b0 + kk * 32),
                          idesc, kk != 0 ? 1u : 0u);
          issued = true;
          ptx::mma_commit(&sm.empty[s]);
          ptx::mma_commit(&sm.pfull[b]);
          if (++s == STAGES) {
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
  } else if (warp == SCALE_WARP) {
    // ======================= scale warp =====================================
    constexpr int CPL = BNMAX / 32;  // token columns per lane
    const int NBk = p.N / 128;       // weight scale blocks along N
    uint32_t kbg = 0;
    bool ok = true;
    for (int g = blockIdx.x; ok && g < total; g += ncta) {
      const TileInfo<BNMAX> t = decode_tile<BNMAX>(sm, E, p.NB, g);
      // the scale blocks of the tile's weight rows: its 128-row block (bf16
      // out), or the block of its 64 gate rows and of its 64 up rows (SiLU)
      const float* sbe = p.scale_b + (int64_t)t.e * NBk * KB;
      const float* sb0 = sbe + (SILU ? t.nb / 2 : t.nb) * KB;
      const float* sb1 = sbe + (SILU ? (p.I + t.nb * 64) / 128 : t.nb) * KB;
      const float* sa_t = p.scale_a + (int64_t)t.tok0 * KB;
      if ((KB & 3) == 0 && ((reinterpret_cast<uintptr_t>(p.scale_a) |
                             reinterpret_cast<uintptr_t>(p.scale_b)) & 15) == 0) {
        // four K blocks of scales per 16-byte load, the next four loaded
        // while these are used
        float4 cur[CPL], nxt[CPL];
        float4 b0c, b1c, b0n, b1n;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int col = c * 32 + lane;
          cur[c] = col < t.ntok ? __ldg(reinterpret_cast<const float4*>(sa_t + col * KB))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        b0c = __ldg(reinterpret_cast<const float4*>(sb0));
        b1c = SILU ? __ldg(reinterpret_cast<const float4*>(sb1)) : b0c;
#pragma unroll
        for (int c = 0; c < CPL; ++c) nxt[c] = cur[c];
        b0n = b0c;
        b1n = b1c;
        if (KB > 4) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int col = c * 32 + lane;
            nxt[c] = col < t.ntok ? __ldg(reinterpret_cast<const float4*>(sa_t + col * KB + 4))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          b0n = __ldg(reinterpret_cast<const float4*>(sb0 + 4));
          b1n = SILU ? __ldg(reinterpret_cast<const float4*>(sb1 + 4)) : b0n;
        }
        for (int kb = 0; kb < KB; ++kb, ++kbg) {
          const int j = kb & 3;
          if (j == 0 && kb > 0) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) cur[c] = nxt[c];
            b0c = b0n;
            b1c = b1n;
            if (kb + 4 < KB) {
#pragma unroll
              for (int c = 0; c < CPL; ++c) {
                const int col = c * 32 + lane;
                nxt[c] = col < t.ntok
                             ? __ldg(reinterpret_cast<const float4*>(sa_t + col * KB + kb + 4))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
              }
              b0n = __ldg(reinterpret_cast<const float4*>(sb0 + kb + 4));
              b1n = SILU ? __ldg(reinterpret_cast<const float4*>(sb1 + kb + 4)) : b0n;
            }
          }
          const uint32_t b = kbg % NPB;
          ok = ptx::mbar_wait(&sm.sempty[b], ((kbg / NPB) & 1u) ^ 1u, &sm.abort, WAIT_NS);
          if (!__all_sync(kFull, ok)) {
            ok = false;
            break;
          }
          const float s0 = j == 0 ? b0c.x : j == 1 ? b0c.y : j == 2 ? b0c.z : b0c.w;
          const float s1 = j == 0 ? b1c.x : j == 1 ? b1c.y : j == 2 ? b1c.z : b1c.w;
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const float a = j == 0 ? cur[c].x : j == 1 ? cur[c].y : j == 2 ? cur[c].z : cur[c].w;
            sm.fs[b][0][c * 32 + lane] = a * s0;
            if (SILU) sm.fs[b][NF - 1][c * 32 + lane] = a * s1;
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.sfull[b]);
        }
        continue;
      }
      float sa[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int col = c * 32 + lane;
        sa[c] = col < t.ntok ? __ldg(sa_t + col * KB) : 0.0f;
      }
      float s0 = __ldg(sb0), s1 = SILU ? __ldg(sb1) : 0.0f;
      for (int kb = 0; kb < KB; ++kb, ++kbg) {
        const uint32_t b = kbg % NPB;
        ok = ptx::mbar_wait(&sm.sempty[b], ((kbg / NPB) & 1u) ^ 1u, &sm.abort, WAIT_NS);
        if (!__all_sync(kFull, ok)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          sm.fs[b][0][c * 32 + lane] = sa[c] * s0;
          if (SILU) sm.fs[b][NF - 1][c * 32 + lane] = sa[c] * s1;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.sfull[b]);
        if (kb + 1 < KB) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int col = c * 32 + lane;
            sa[c] = col < t.ntok ? __ldg(sa_t + col * KB + kb + 1) : 0.0f;
          }
          s0 = __ldg(sb0 + kb + 1);
          if (SILU) s1 = __ldg(sb1 + kb + 1);
        }
      }
    }
    if (!ok && lane == 0) {
      sm.abort = 1;
      flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
    }
  } else {
    // ======================= epilogue (warps 2 .. 2 + EW - 1) ===============
    const int ew = warp - 2;
    const int q = warp & 3;                   // TMEM lane quadrant this warp may access
    const int cg = ew >> 2;                   // column group: chunks cg, cg + CG, ...
    const int frow = SILU && q >= 2 ? 1 : 0;  // factor row: up rows (SiLU) or the block
    uint32_t kbg = 0;
    bool stop = false;
    for (int g = blockIdx.x; !stop && g < total; g += ncta) {
      const TileInfo<BNMAX> t = decode_tile<BNMAX>(sm, E, p.NB, g);
      const int n_mma = (t.ntok + 15) & ~15;
      float acc[HC];
#pragma unroll
      for (int i = 0; i < HC; ++i) acc[i] = 0.0f;
      for (int kb = 0; kb < KB; ++kb, ++kbg) {
        const uint32_t b = kbg % NPB;
        const uint32_t par = (kbg / NPB) & 1u;
        bool ok = ptx::mbar_wait(&sm.pfull[b], par, &sm.abort, WAIT_NS) &&
                  ptx::mbar_wait(&sm.sfull[b], par, &sm.abort, WAIT_NS);
        if (!__all_sync(kFull, ok)) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + b * BNMAX;
        const float* fr = sm.fs[b][frow];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int col0 = (cg + c * CG) * 32;
          if (col0 < n_mma) {  // warp-uniform
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tb + col0, v);
            ptx::tmem_ld_wait();
            ptx::reg_fence(v);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 fv = *reinterpret_cast<const float4*>(fr + col0 + i);
              float* a = acc + c * 32 + i;
              fma2(a[0], a[1], __uint_as_float(v[i + 0]), __uint_as_float(v[i + 1]), fv.x, fv.y);
              fma2(a[2], a[3], __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]), fv.z, fv.w);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&sm.pempty[b]);
          ptx::mbar_arrive(&sm.sempty[b]);
        }
      }
      // the two warps of a SiLU exchange pair go on to the output together
      // or not at all (a warp that stopped still meets its partner here)
      if (SILU && bar_red_or(BAR_PAIR + (q & 1) + 2 * cg, 64, stop)) stop = true;
      if (stop) break;
      // ---- the tile's output: every K block is in acc ----
      if (SILU) {
        const int I = p.I;
        const int pair = (q & 1) + 2 * cg;
        const bool holds_gate = q < 2;
        const int mine0 = holds_gate ? 0 : 16;  // gate: tokens 0..15 of a chunk, up: 16..31
        // this warp gives through its own slot and reads its partner's (the
        // warp of the other lane half, same column group)
        float* give = reinterpret_cast<float*>(sm.scr[ew]);
        float* take = reinterpret_cast<float*>(sm.scr[ew ^ 2]);
        uint16_t* ost = reinterpret_cast<uint16_t*>(take);
        const int jrow = t.nb * 64 + (q & 1) * 32;  // first j of this warp's 32
        __nv_bfloat16* hbase = reinterpret_cast<__nv_bfloat16*>(p.C);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int col0 = (cg + c * CG) * 32;  // first token column of the chunk
          if (col0 >= t.ntok) break;            // the same for both warps of the pair
          // the gate holder gives tokens 16..31, the up holder tokens 0..15
#pragma unroll
          for (int i = 0; i < 16; ++i)
            give[i * 32 + lane] = holds_gate ? acc[c * 32 + 16 + i] : acc[c * 32 + i];
          bar_sync_named(BAR_PAIR + pair, 64);
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float own = holds_gate ? acc[c * 32 + i] : acc[c * 32 + 16 + i];
            const float other = take[i * 32 + lane];
            const float gv = holds_gate ? own : other;
            const float uv = holds_gate ? other : own;
            hv[i] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
          }
          __syncwarp();  // the partner's values are read: its slot takes the bf16 rows
#pragma unroll
          for (int i = 0; i < 16; ++i)
            ost[i * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(hv[i]));
          __syncwarp();
          // 16 tokens x 32 j: four lanes per token row, 16 bytes each
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int r = k * 8 + (lane >> 2);
            const int tk = col0 + mine0 + r;
            if (tk < t.ntok)
              *reinterpret_cast<uint4*>(hbase + (int64_t)(t.tok0 + tk) * I + jrow +
                                        (lane & 3) * 8) =
                  *reinterpret_cast<const uint4*>(ost + r * 32 + (lane & 3) * 8);
          }
          __syncwarp();
          bar_sync_named(BAR_PAIR + pair, 64);  // both slots are free again
        }
      } else {
        const int N = p.N;
        const int ncol0 = t.nb * BM + q * 32;  // first output column of this warp's 32
        uint16_t* ost = reinterpret_cast<uint16_t*>(sm.scr[ew]);
        __nv_bfloat16* cbase = reinterpret_cast<__nv_bfloat16*>(p.C);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int col0 = (cg + c * CG) * 32;
          if (col0 >= t.ntok) break;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            ost[i * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[c * 32 + i]));
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int r = k * 8 + (lane >> 2);
            if (col0 + r < t.ntok)
              *reinterpret_cast<uint4*>(cbase + (int64_t)(t.tok0 + col0 + r) * N + ncol0 +
                                        (lane & 3) * 8) =
                  *reinterpret_cast<const uint4*>(ost + r * 32 + (lane & 3) * 8);
          }
          __syncwarp();
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
    for (int i = 0; i < STAGES; ++i)
      if ((armed >> i) & 1u)
        ptx::mbar_wait(&sm.full[i], (armed_par >> i) & 1u, &sm.never, DRAIN_NS);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TCOLS);
  }
}

// The deepest ring that fits next to the rest of the shared memory (at most 8).
template <int BNMAX, int NF>
constexpr int block_stages() {
  constexpr size_t per = W_BYTES + BNMAX * BK + 16;
  constexpr size_t fixed = sizeof(BSmem<BNMAX, 1, NF>) - per + 16 + 1024;
  constexpr size_t n = (227 * 1024 - fixed) / per;
  return n > 8 ? 8 : (int)n;
}

template <int BNMAX, bool SILU>
cudaError_t launch_block_cfg(const Maps& maps, const BParams& p, int M, int E, cudaStream_t st,
                             bool pdl) {
  constexpr int NF = SILU ? 2 : 1;
  constexpr int STAGES = block_stages<BNMAX, NF>();
  static_assert(STAGES >= 3, "pipeline depth");
  constexpr size_t smem = sizeof(BSmem<BNMAX, STAGES, NF>) + 1024;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = grouped_gemm_block_kernel<BNMAX, STAGES, SILU>;
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
  const long long upper = ((long long)(M + BNMAX - 1) / BNMAX + E) * p.NB;
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
  // one K block per stage: weight boxes of one chunk (Kd % 128 == 0, checked
  // at the entry point, keeps the chunked weight view inside the tensor)
  Maps maps;
  if (!weights_stage_box((uint64_t)Kd) ||
      !make_tma_map_weights(&maps.w, B, silu, (uint64_t)E, (uint64_t)N, (uint64_t)Kd, 1))
    return cudaErrorNotSupported;
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
  if (small)
    return silu ? launch_block_cfg<64, true>(maps, p, M, E, st, pdl)
                : launch_block_cfg<64, false>(maps, p, M, E, st, pdl);
  return silu ? launch_block_cfg<128, true>(maps, p, M, E, st, pdl)
              : launch_block_cfg<128, false>(maps, p, M, E, st, pdl);
}

}  // namespace moe
