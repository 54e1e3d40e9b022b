// moe_grouped_gemm: FP8 (e4m3) grouped GEMM over expert row segments on the
// 5th-generation tensor cores, with the per-row x per-channel dequantisation
// fused into the epilogue ("Fix one bug in the grouped-gemm triton kernel",
// sglang #6772, Highlights: scale_a is indexed by the row, m_range_start +
// offs_am; "Support token-level quantization for EP MoE", sglang #6782,
// Changelog: per-token scale_a in the grouped GEMM).
//
// Design (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0      TMA producer: A tile [128 rows x 128 B] + B tile
//               [256 rows x 128 B] per stage into a 4-stage ring, 128-byte
//               swizzled; weights streamed with an evict-first L2 policy,
//               activations kept with evict-last.
//   warp 1      MMA issuer: tcgen05.mma.cta_group::1.kind::f8f6f4,
//               M=128 x N=256 x K=32 per instruction, fp32 accumulator in
//               tensor memory; two accumulators (2 x 256 columns) so the
//               epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one token row per
//               thread), dequantise by scale_a[row] * scale_b[e,n], then
//               either bf16 out or SiLU(gate) * up -> bf16 (+ row amax).
// Tiles are (expert, n-block, m-block) with the m-block fastest, so the
// m-blocks of one expert stream the same weight block at the same time and
// share it through L2. The tile table is derived on the device from the
// expert offsets (no host synchronisation); rows of a tile past the
// expert's segment are computed but never stored.
// For SiLU*mul, the n-block takes gate rows [nb*128, nb*128+128) and the
// matching up rows [I+nb*128, ...) as the two halves of the 256-row B tile,
// so gate and up land in the same thread's accumulator columns.
// Every pipeline wait is bounded (2 s); on timeout the CTA sets the device
// error word, lets its in-flight copies and MMAs land, frees its tensor
// memory and exits.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;   // token rows per tile (MMA M)
constexpr int BN = 256;   // weight rows per tile (MMA N)
constexpr int BK = 128;   // K bytes (= e4m3 elements) per pipeline stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int MAX_E = 1024;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_NS = 200000000ull;

struct Smem {
  uint8_t a[STAGES][A_BYTES];  // each stage 1024-byte aligned (swizzle atom)
  uint8_t b[STAGES][B_BYTES];
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
  int M, N, Kd, E, epilogue, I, NB, KB;
};

// tile -> (expert, n-block, m-block)
__device__ __forceinline__ void decode_tile(const Smem& sm, int E, int NB, int tile, int& e,
                                            int& nb, int& mb) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  const int local = tile - sm.tile_start[e];
  const int mbc = (sm.tile_start[e + 1] - sm.tile_start[e]) / NB;
  nb = local / mbc;
  mb = local - nb * mbc;
}

__device__ __forceinline__ void load_scales32(const float* p, int valid_cols, float (&s)[32]) {
  if (valid_cols >= 32) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p + i));
      s[i] = v.x;
      s[i + 1] = v.y;
      s[i + 2] = v.z;
      s[i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = (i < valid_cols) ? __ldg(p + i) : 0.0f;
  }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const uint32_t (&pk)[16],
                                              int valid_cols) {
  if (valid_cols >= 32) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      d[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  } else {
    uint16_t* d = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < valid_cols) d[i] = (uint16_t)((i & 1) ? (pk[i >> 1] >> 16) : (pk[i >> 1] & 0xffffu));
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sm.tfull[b], 1);
      ptx::mbar_init(&sm.tempty[b], 128);
    }
    ptx::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    sm.never = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }

  // ---- tile table from the expert offsets --------------------------------
  for (int i = tid; i <= E; i += THREADS) sm.offs[i] = __ldg(p.offsets + i);
  __syncthreads();
  const int per = (E + THREADS - 1) / THREADS;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  int bad = 0;
  for (int e = e0; e < e1; ++e) {
    const int lo = sm.offs[e], hi = sm.offs[e + 1];
    if (lo < 0 || hi < lo || hi > p.M) bad = 1;
    else local += (hi - lo + BM - 1) / BM;
  }
  sm.thr_sum[tid] = local;
  bad = __syncthreads_or(bad);
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < THREADS; ++i) {
      const int v = sm.thr_sum[i];
      sm.thr_sum[i] = run;
      run += v;
    }
    sm.total_tiles = bad ? 0 : run * p.NB;
    sm.tile_start[E] = run * p.NB;
    if (bad) flag_error(p.err, MOE_DEV_BAD_OFFSETS);
  }
  __syncthreads();
  {
    int run = sm.thr_sum[tid];
    for (int e = e0; e < e1; ++e) {
      sm.tile_start[e] = run * p.NB;
      const int lo = sm.offs[e], hi = sm.offs[e + 1];
      if (!bad) run += (hi - lo + BM - 1) / BM;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int total = sm.total_tiles;

  if (warp == 0) {
    // ======================= TMA producer ===================================
    if (lane == 0) {
      const uint64_t pol_a = ptx::policy_evict_last();
      const uint64_t pol_b = ptx::policy_evict_first();
      uint32_t s = 0, ph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, nb, mb;
        decode_tile(sm, E, p.NB, tile, e, nb, mb);
        const int m0 = sm.offs[e] + mb * BM;
        int y0, y1;
        if (p.epilogue == MOE_EPI_SILU_MUL) {
          y0 = e * p.N + nb * 128;
          y1 = y0 + p.I;
        } else {
          y0 = e * p.N + nb * BN;
          y1 = y0 + 128;
        }
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!ptx::mbar_wait(&sm.empty[s], ph ^ 1u, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&sm.full[s], STAGE_BYTES);
          armed |= 1u << s;
          armed_par = (armed_par & ~(1u << s)) | (ph << s);
          ptx::tma_load_2d(sm.a[s], &tmA, &sm.full[s], kb * BK, m0, pol_a);
          ptx::tma_load_2d(sm.b[s], &tmB, &sm.full[s], kb * BK, y0, pol_b);
          ptx::tma_load_2d(sm.b[s] + 128 * BK, &tmB, &sm.full[s], kb * BK, y1, pol_b);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        for (int i = 0; i < STAGES; ++i)
          if ((armed >> i) & 1u)
            ptx::mbar_wait(&sm.full[i], (armed_par >> i) & 1u, &sm.never, DRAIN_NS);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =====================================
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_e4m3_f32(BM, BN);
      uint32_t s = 0, ph = 0;
      bool ok = true, issued = false;
      int iter = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++iter) {
        const int b = iter & 1;
        const uint32_t tph = (iter >> 1) & 1;
        if (!ptx::mbar_wait(&sm.tempty[b], tph ^ 1u, &sm.abort, WAIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * BN);
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!ptx::mbar_wait(&sm.full[s], ph, &sm.abort, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sm.a[s]);
          const uint32_t b0 = ptx::smem_u32(sm.b[s]);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            ptx::mma_e4m3(d, ptx::sdesc_sw128(a0 + kk * 32), ptx::sdesc_sw128(b0 + kk * 32),
                          idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          issued = true;
          ptx::mma_commit(&sm.empty[s]);
          if (++s == STAGES) {
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
  } else {
    // ======================= epilogue (warps 2..5) ==========================
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int iter = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++iter) {
      const int b = iter & 1;
      const uint32_t tph = (iter >> 1) & 1;
      int e, nb, mb;
      decode_tile(sm, E, p.NB, tile, e, nb, mb);
      const int row = sm.offs[e] + mb * BM + q * 32 + lane;
      const bool valid = row < sm.offs[e + 1];
      bool ok = ptx::mbar_wait(&sm.tfull[b], tph, &sm.abort, WAIT_NS);
      ok = __all_sync(kFull, ok);
      if (!ok) {
        sm.abort = 1;
        flag_error(p.err, MOE_DEV_PIPE_TIMEOUT);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN);
      const float sa = valid ? __ldg(p.scale_a + row) : 0.0f;
      if (p.epilogue == MOE_EPI_SILU_MUL) {
        const int I = p.I;
        __nv_bfloat16* hrow = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * I;
        float amax = 0.0f;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32x32b_x32(tbase + c, g);
          ptx::tmem_ld_32x32b_x32(tbase + 128 + c, u);
          ptx::tmem_ld_wait();
          ptx::reg_fence(g);
          ptx::reg_fence(u);
          const int j0 = nb * 128 + c;
          const int vc = min(32, I - j0);
          if (!valid || vc <= 0) continue;
          float sg[32], su[32];
          const float* sb = p.scale_b + (int64_t)e * p.N + j0;
          load_scales32(sb, vc, sg);
          load_scales32(sb + I, vc, su);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float hv[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float gv = __uint_as_float(g[i + h]) * sa * sg[i + h];
              const float uv = __uint_as_float(u[i + h]) * sa * su[i + h];
              hv[h] = gv / (1.0f + __expf(-gv)) * uv;
            }
            pk[i >> 1] = pack_bf16x2(hv[0], hv[1]);
            const float r0 = fabsf(__uint_as_float(pk[i >> 1] << 16));
            const float r1 = fabsf(__uint_as_float(pk[i >> 1] & 0xffff0000u));
            if (i < vc) amax = fmaxf(amax, r0);
            if (i + 1 < vc) amax = fmaxf(amax, r1);
          }
          store_bf16x32(hrow + j0, pk, vc);
        }
        if (p.row_amax != nullptr && valid)
          atomicMax(reinterpret_cast<int*>(p.row_amax + row), __float_as_int(amax));
      } else {
        const int N = p.N;
        __nv_bfloat16* crow = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * N;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t acc[32];
          ptx::tmem_ld_32x32b_x32(tbase + c, acc);
          ptx::tmem_ld_wait();
          ptx::reg_fence(acc);
          const int n0 = nb * BN + c;
          const int vc = min(32, N - n0);
          if (!valid || vc <= 0) continue;
          float sb[32];
          load_scales32(p.scale_b + (int64_t)e * N + n0, vc, sb);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            pk[i >> 1] = pack_bf16x2(__uint_as_float(acc[i]) * sa * sb[i],
                                     __uint_as_float(acc[i + 1]) * sa * sb[i + 1]);
          store_bf16x32(crow + n0, pk, vc);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.tempty[b]);
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- host side ---------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D u8 tensor [rows, cols] (cols contiguous), box 128 x 128, 128-byte
// swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {BK, 128};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

}  // namespace

cudaError_t launch_grouped_gemm(const void* A, const float* scale_a, const void* B,
                                const float* scale_b, const int32_t* offsets, int M, int N,
                                int Kd, int E, int epilogue, void* C, float* row_amax, int* err,
                                cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  if (!make_map(&mA, A, (uint64_t)M, (uint64_t)Kd) ||
      !make_map(&mB, B, (uint64_t)E * (uint64_t)N, (uint64_t)Kd))
    return cudaErrorNotSupported;
  Params p;
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
  p.epilogue = epilogue;
  p.I = N / 2;
  p.NB = (epilogue == MOE_EPI_SILU_MUL) ? (p.I + 127) / 128 : (N + BN - 1) / BN;
  p.KB = (Kd + BK - 1) / BK;
  const long long upper = ((long long)(M + BM - 1) / BM + E) * p.NB;
  const int grid = (int)std::min<long long>(sm_count(), upper);

  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 64 || !attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
      if (e != cudaSuccess) return e;
      if (dev < 64) attr_set[dev] = true;
    }
  }
  grouped_gemm_kernel<<<grid, THREADS, kSmemBytes, st>>>(mA, mB, p);
  return cudaGetLastError();
}

}  // namespace moe
