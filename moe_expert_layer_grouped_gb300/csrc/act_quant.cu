// moe_act_quant: per-token FP8 requantisation of the SiLU*mul output
// ("Support token-level quantization for EP MoE", sglang #6782, Changelog
// and Code Review: down_input is requantised per token, giving
// w2_input_scale). 128-bit loads; a row is read from memory once: it stays
// in registers between its amax and its codes (one warp per row up to 512
// channels, one CTA per row up to 16384). Longer rows, and rows whose amax
// the caller supplies, take one warp per row in two passes (the amax,
// skipped when supplied, then the codes). The block variant (one
// scale per 128 channels, the block-quantised FP8 path) quantises each block
// in one pass.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    act_quant_kernel(const __nv_bfloat16* __restrict__ h, const float* __restrict__ row_amax,
                     int M, int I, uint8_t* __restrict__ q, float* __restrict__ scale) {
  chain_entry();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  if (row >= M) return;
  const int nvec = I >> 3;
  const uint4* hr = reinterpret_cast<const uint4*>(h + row * I);
  float amax;
  if (row_amax != nullptr) {
    amax = __ldg(row_amax + row);
  } else {
    amax = 0.0f;
#pragma unroll 4
    for (int i = lane; i < nvec; i += 32) {
      float f[8];
      bf16x8_to_f32(__ldg(hr + i), f);
      amax = absmax8(f, amax);
    }
    amax = warp_max(amax);
  }
  const float sc = token_scale(amax);
  if (lane == 0) scale[row] = sc;
  const Recip rb = recip_bracket(sc);
  uint2* qr = reinterpret_cast<uint2*>(q + row * I);
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) {
    float f[8];
    bf16x8_to_f32(__ldg(hr + i), f);
    qr[i] = quant8(f, rb);
  }
}

// One row in registers: vector u * NT + tid of the row in raw[u] (NT threads
// per row: a warp, or a CTA with `red` holding its warps' maxima).
template <int V, int NT>
__device__ __forceinline__ void quant_row_in_regs(const uint4* __restrict__ hr, int nvec, int tid,
                                                  float* red, uint2* __restrict__ qr,
                                                  float* __restrict__ scale_out) {
  uint4 raw[V];
  float amax = 0.0f;
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int i = u * NT + tid;
    if (i < nvec) {
      raw[u] = __ldg(hr + i);
      float f[8];
      bf16x8_to_f32(raw[u], f);
      amax = absmax8(f, amax);
    }
  }
  amax = warp_max(amax);
  if constexpr (NT > 32) {
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) amax = fmaxf(amax, red[w]);
  }
  const float sc = token_scale(amax);
  if (tid == 0) *scale_out = sc;
  const Recip rb = recip_bracket(sc);
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int i = u * NT + tid;
    if (i < nvec) {
      float f[8];
      bf16x8_to_f32(raw[u], f);
      qr[i] = quant8(f, rb);
    }
  }
}

template <int V>  // vectors per lane: rows of up to 256 V channels
__global__ void __launch_bounds__(kWarps * 32)
    act_quant_warp_kernel(const __nv_bfloat16* __restrict__ h, int M, int I,
                          uint8_t* __restrict__ q, float* __restrict__ scale) {
  chain_entry();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  if (row >= M) return;  // warp-uniform
  quant_row_in_regs<V, 32>(reinterpret_cast<const uint4*>(h + row * I), I >> 3, lane, nullptr,
                           reinterpret_cast<uint2*>(q + row * I), scale + row);
}

template <int V, int NT>  // vectors per thread, threads: rows of up to 8 V NT channels
__global__ void __launch_bounds__(NT)
    act_quant_cta_kernel(const __nv_bfloat16* __restrict__ h, int I, uint8_t* __restrict__ q,
                         float* __restrict__ scale) {
  chain_entry();
  __shared__ float red[NT / 32];
  const int64_t row = blockIdx.x;
  quant_row_in_regs<V, NT>(reinterpret_cast<const uint4*>(h + row * I), I >> 3, threadIdx.x,
                           red, reinterpret_cast<uint2*>(q + row * I), scale + row);
}

// Block requantisation: one scale per 128 channels of a row (scale
// [M, I/128]). A warp takes a row two blocks at a time, a half-warp per
// block (16 lanes x 8 values), the block amax by a 16-lane shuffle; the
// loads of four such steps are issued before the first is used.
__global__ void __launch_bounds__(kWarps * 32)
    act_quant_block_kernel(const __nv_bfloat16* __restrict__ h, int M, int I,
                           uint8_t* __restrict__ q, float* __restrict__ scale) {
  chain_entry();
  constexpr int U = 4;  // steps of two blocks in flight
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  if (row >= M) return;  // warp-uniform
  const int nb = I >> 7;
  const uint4* hr = reinterpret_cast<const uint4*>(h + row * I);
  uint2* qr = reinterpret_cast<uint2*>(q + row * I);
  for (int b0 = 0; b0 < nb; b0 += 2 * U) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int b = b0 + 2 * u + (lane >> 4);
      if (b < nb) raw[u] = __ldg(hr + b * 16 + (lane & 15));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int b = b0 + 2 * u + (lane >> 4);
      const bool in = b < nb;
      float f[8];
      float m = 0.0f;
      if (in) {
        bf16x8_to_f32(raw[u], f);
        m = absmax8(f, 0.0f);
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      if (in) {
        const float sc = token_scale(m);
        qr[b * 16 + (lane & 15)] = quant8(f, sc);
        if ((lane & 15) == 0) scale[row * nb + b] = sc;
      }
    }
  }
}

// NVFP4 requantisation of h with the global scale g: q [M, I/2] (two E2M1
// codes per byte), sf [M, I/16] E4M3 block scales. One warp per row; a
// 16-channel block is the 8-value vectors of lanes 2i and 2i+1.
__global__ void __launch_bounds__(kWarps * 32)
    act_quant_nvfp4_kernel(const __nv_bfloat16* __restrict__ h, int M, int I, float g,
                           uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  chain_entry();
  constexpr int U = 4;  // vectors per lane in flight
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  if (row >= M) return;  // warp-uniform
  const int nvec = I >> 3;
  const uint4* hr = reinterpret_cast<const uint4*>(h + row * I);
  uint32_t* qr = reinterpret_cast<uint32_t*>(q + row * (I >> 1));
  uint8_t* sr = sf + row * (I >> 4);
  const Recip rg = recip_bracket(g);
  for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = v0 + u * 32 + lane;
      if (i < nvec) raw[u] = __ldg(hr + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = v0 + u * 32 + lane;
      float f[8];
      float m = 0.0f;
      if (i < nvec) {
        bf16x8_to_f32(raw[u], f);
        m = absmax8(f, 0.0f);
      }
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
      if (i < nvec) {
        const uint32_t code = nvfp4_scale_code(m, g, rg);
        qr[i] = nvfp4_codes8(f, __fmul_rn(e4m3_value(code), g));
        if ((i & 1) == 0) sr[i >> 1] = (uint8_t)code;
      }
    }
  }
}

// The same with a row per CTA, read once (as the FP8 requant): vector
// u * NT + tid in registers, every load of the row issued before the first
// is used; each eighth thread stores the scale bytes of four blocks (its own
// and those of the threads 2, 4 and 6 above it) as one word.
template <int V, int NT>
__global__ void __launch_bounds__(NT)
    act_quant_nvfp4_cta_kernel(const __nv_bfloat16* __restrict__ h, int I, float g,
                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  chain_entry();
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int nvec = I >> 3;  // I % 256 == 0: a multiple of 32, validity is warp-uniform
  const uint4* hr = reinterpret_cast<const uint4*>(h + row * I);
  uint32_t* qr = reinterpret_cast<uint32_t*>(q + row * (I >> 1));
  uint8_t* sr = sf + row * (I >> 4);
  const Recip rg = recip_bracket(g);
  uint4 raw[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int i = u * NT + tid;
    if (i < nvec) raw[u] = __ldg(hr + i);
  }
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int i = u * NT + tid;
    if (i >= nvec) break;  // warp-uniform
    float f[8];
    bf16x8_to_f32(raw[u], f);
    float m = absmax8(f, 0.0f);
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
    const uint32_t code = nvfp4_scale_code(m, g, rg);
    qr[i] = nvfp4_codes8(f, __fmul_rn(e4m3_value(code), g));
    const uint32_t c2 = __shfl_down_sync(kFull, code, 2);
    const uint32_t c4 = __shfl_down_sync(kFull, code, 4);
    const uint32_t c6 = __shfl_down_sync(kFull, code, 6);
    if ((tid & 7) == 0)
      *reinterpret_cast<uint32_t*>(sr + (i >> 1)) = code | (c2 << 8) | (c4 << 16) | (c6 << 24);
  }
}

}  // namespace

cudaError_t launch_act_quant_nvfp4(const void* h, int M, int I, float g, void* q, uint8_t* sf,
                                   cudaStream_t st, bool pdl) {
  if (M == 0) return cudaSuccess;
  // a row per CTA held in registers up to 16384 channels (65536 x 2048:
  // 64 threads of 4 vectors) when I % 256 == 0 (whole warps of vectors, and
  // 4-byte-aligned words of scale bytes); a warp per row in steps of 4
  // vectors a lane otherwise
  const int nvec = I >> 3;
  const __nv_bfloat16* hb = reinterpret_cast<const __nv_bfloat16*>(h);
  uint8_t* qb = reinterpret_cast<uint8_t*>(q);
#define MOE_AQF(V, NT) launch_kernel(act_quant_nvfp4_cta_kernel<V, NT>, dim3(M), dim3(NT), 0, \
                                     st, pdl, hb, I, g, qb, sf)
  if (I % 256 == 0) {
    if (nvec <= 64 * 2) return MOE_AQF(2, 64);
    if (nvec <= 64 * 4) return MOE_AQF(4, 64);
    if (nvec <= 256 * 2) return MOE_AQF(2, 256);
    if (nvec <= 256 * 4) return MOE_AQF(4, 256);
    if (nvec <= 256 * 6) return MOE_AQF(6, 256);
    if (nvec <= 256 * 8) return MOE_AQF(8, 256);
  }
#undef MOE_AQF
  const int blocks = (M + kWarps - 1) / kWarps;
  return launch_kernel(act_quant_nvfp4_kernel, dim3(blocks), dim3(kWarps * 32), 0, st, pdl,
                       reinterpret_cast<const __nv_bfloat16*>(h), M, I, g,
                       reinterpret_cast<uint8_t*>(q), sf);
}

cudaError_t launch_act_quant_block(const void* h, int M, int I, void* q, float* scale,
                                   cudaStream_t st, bool pdl) {
  if (M == 0) return cudaSuccess;
  const int blocks = (M + kWarps - 1) / kWarps;
  return launch_kernel(act_quant_block_kernel, dim3(blocks), dim3(kWarps * 32), 0, st, pdl,
                       reinterpret_cast<const __nv_bfloat16*>(h), M, I,
                       reinterpret_cast<uint8_t*>(q), scale);
}

cudaError_t launch_act_quant(const void* h, const float* row_amax, int M, int I, void* q,
                             float* scale, cudaStream_t st, bool pdl) {
  if (M == 0) return cudaSuccess;
  const int blocks = (M + kWarps - 1) / kWarps;
  const int nvec = I >> 3;
  const __nv_bfloat16* hb = reinterpret_cast<const __nv_bfloat16*>(h);
  uint8_t* qb = reinterpret_cast<uint8_t*>(q);
  // Rows of up to 512 channels: a warp per row. Longer ones: a CTA per row,
  // 64 threads up to 2048 channels (a 2048-channel row: 70.7 us for 65536
  // rows, against 76 us with a warp per row holding 8 vectors a lane and
  // 101 us in two passes), 256 threads up to 16384.
  if (row_amax == nullptr && nvec <= 64) {
    if (nvec <= 32)
      return launch_kernel(act_quant_warp_kernel<1>, dim3(blocks), dim3(kWarps * 32), 0, st, pdl,
                           hb, M, I, qb, scale);
    return launch_kernel(act_quant_warp_kernel<2>, dim3(blocks), dim3(kWarps * 32), 0, st, pdl,
                         hb, M, I, qb, scale);
  }
  if (row_amax == nullptr && nvec <= 256 * 8) {
#define MOE_AQC(V, NT) launch_kernel(act_quant_cta_kernel<V, NT>, dim3(M), dim3(NT), 0, st, \
                                     pdl, hb, I, qb, scale)
    if (nvec <= 64 * 2) return MOE_AQC(2, 64);
    if (nvec <= 64 * 4) return MOE_AQC(4, 64);
    if (nvec <= 256 * 2) return MOE_AQC(2, 256);
    if (nvec <= 256 * 4) return MOE_AQC(4, 256);
    if (nvec <= 256 * 6) return MOE_AQC(6, 256);
    return MOE_AQC(8, 256);
#undef MOE_AQC
  }
  return launch_kernel(act_quant_kernel, dim3(blocks), dim3(kWarps * 32), 0, st, pdl,
                       reinterpret_cast<const __nv_bfloat16*>(h), row_amax, M, I,
                       reinterpret_cast<uint8_t*>(q), scale);
}

}  // namespace moe
