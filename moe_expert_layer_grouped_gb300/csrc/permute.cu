// moe_permute_quant: pre-reorder with dynamic per-token FP8 quantisation
// ("Support token-level quantization for EP MoE", sglang #6782, Summary of
// Changes / Changelog / Code Review; expert row ranges from "Fix one bug in
// the grouped-gemm triton kernel", sglang #6772, Highlights).
//
// Three launches, all deterministic (no atomics whose order matters):
//  1. route_bits: for every block of 32 tokens c and expert e, a 32-bit mask
//     of the tokens in the block that chose e (bits[c][e]).
//  2. route_scan (one CTA): per expert, the running token count before each
//     block (base[c][e], absolute row index) and the offsets table.
//  3. permute_quant (one CTA per token): the token's K destination rows are
//     base[c][e] + popcount(bits[c][e] below the token's bit) -- a stable
//     counting sort by expert in ascending token order -- and its row is
//     loaded once (128-bit vectors, kept in registers), reduced to amax,
//     quantised and stored to all K destinations with its scale.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kBitsWarps = 8;

__global__ void __launch_bounds__(kBitsWarps * 32)
    route_bits_kernel(const int32_t* __restrict__ ids, int T, int E, int K,
                      uint32_t* __restrict__ bits, int* err) {
  extern __shared__ uint32_t masks[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = (T + 31) >> 5;
  const int c = blockIdx.x * kBitsWarps + warp;
  if (c >= C) return;  // warp-uniform
  uint32_t* my = masks + warp * E;
  for (int e = lane; e < E; e += 32) my[e] = 0u;
  __syncwarp();
  const int t = c * 32 + lane;
  if (t < T) {
    const int32_t* row = ids + (int64_t)t * K;
    for (int k = 0; k < K; ++k) {
      const int e = row[k];
      bool ok = (unsigned)e < (unsigned)E;
      for (int j = 0; j < k && ok; ++j) ok = (row[j] != e);  // distinct per token
      if (ok)
        atomicOr(&my[e], 1u << lane);
      else
        flag_error(err, MOE_DEV_BAD_EXPERT_ID);
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) bits[(int64_t)c * E + e] = my[e];
}

__global__ void __launch_bounds__(1024)
    route_scan_kernel(const uint32_t* __restrict__ bits, int C, int E,
                      int32_t* __restrict__ base, int32_t* __restrict__ offsets) {
  __shared__ int part[1024];
  __shared__ int total[1024];
  __shared__ int excl[1024];
  __shared__ int warp_sum[32];
  const int tid = threadIdx.x;
  const int P = (E >= 1024) ? 1 : 1024 / E;  // threads per expert
  const int p = tid / E, e = tid % E;
  const bool active = p < P;
  const int per = (C + P - 1) / P;
  const int c0 = min(C, p * per), c1 = min(C, c0 + per);

  int sum = 0;
  if (active)
    for (int c = c0; c < c1; ++c) sum += __popc(__ldg(bits + (int64_t)c * E + e));
  if (active) part[tid] = sum;
  __syncthreads();
  if (tid < E) {
    int run = 0;
    for (int q = 0; q < P; ++q) {
      const int v = part[q * E + tid];
      part[q * E + tid] = run;
      run += v;
    }
    total[tid] = run;
  }
  __syncthreads();
  // exclusive scan of total[0..E) over the block
  const int v = (tid < E) ? total[tid] : 0;
  int incl = v;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int ws = warp_sum[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sum[lane] = wi - ws;  // exclusive prefix of warp totals
  }
  __syncthreads();
  excl[tid] = incl - v + warp_sum[warp];
  if (tid < E) offsets[tid] = excl[tid];
  if (tid == E - 1) offsets[E] = excl[tid] + v;
  __syncthreads();
  if (active) {
    int run = excl[e] + part[tid];
    for (int c = c0; c < c1; ++c) {
      const int64_t i = (int64_t)c * E + e;
      base[i] = run;
      run += __popc(__ldg(bits + i));
    }
  }
}

constexpr int kQuantThreads = 128;

// BLOCK: one scale per 128 channels (scale_a [M, H/128]) instead of one per
// token. A 128-channel block is 16 vectors, held by the 16 lanes of a
// half-warp (vector tid + i*128 lies in block tid/16 + 8i), so its amax is a
// 16-lane shuffle reduction.
template <int VPT, bool BLOCK>  // VPT: 16-byte vectors (8 bf16) per thread
__global__ void __launch_bounds__(kQuantThreads)
    permute_quant_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ ids,
                         const uint32_t* __restrict__ bits, const int32_t* __restrict__ base,
                         int H, int E, int K, uint8_t* __restrict__ a_q,
                         float* __restrict__ scale_a, int32_t* __restrict__ src2dst) {
  __shared__ int dst[32];
  __shared__ float red[kQuantThreads / 32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < K) {
    const int e = __ldg(ids + (int64_t)t * K + tid);
    int d = -1;
    if ((unsigned)e < (unsigned)E) {
      const int64_t i = (int64_t)(t >> 5) * E + e;
      const uint32_t below = __ldg(bits + i) & ((1u << (t & 31)) - 1u);
      d = __ldg(base + i) + __popc(below);
    }
    dst[tid] = d;
    src2dst[(int64_t)t * K + tid] = d;
  }
  const int nvec = H >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)t * H);
  uint4 v[VPT];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = tid + i * kQuantThreads;
    if (idx < nvec) {
      v[i] = __ldg(xr + idx);
      float f[8];
      bf16x8_to_f32(v[i], f);
      amax = absmax8(f, amax);
    }
  }
  if (BLOCK) {
    __syncthreads();  // dst[] is complete
    const int nb = H >> 7;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int idx = tid + i * kQuantThreads;
      float f[8];
      float m = 0.0f;
      if (idx < nvec) {
        bf16x8_to_f32(v[i], f);
        m = absmax8(f, 0.0f);
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      if (idx < nvec) {
        const float sc = token_scale(m);
        const uint2 q = quant8(f, sc);
        for (int k = 0; k < K; ++k) {
          const int d = dst[k];
          if (d < 0) continue;
          *reinterpret_cast<uint2*>(a_q + (int64_t)d * H + (int64_t)idx * 8) = q;
          if ((idx & 15) == 0) scale_a[(int64_t)d * nb + (idx >> 4)] = sc;
        }
      }
    }
    return;
  }
  amax = warp_max(amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float sc = token_scale(amax);
  if (tid < K && dst[tid] >= 0) scale_a[dst[tid]] = sc;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = tid + i * kQuantThreads;
    if (idx < nvec) {
      float f[8];
      bf16x8_to_f32(v[i], f);
      const uint2 q = quant8(f, sc);
      for (int k = 0; k < K; ++k) {
        const int d = dst[k];
        if (d >= 0) *reinterpret_cast<uint2*>(a_q + (int64_t)d * H + (int64_t)idx * 8) = q;
      }
    }
  }
}

template <int VPT, bool BLOCK>
void launch_quant(const void* x, const int32_t* ids, const uint32_t* bits, const int32_t* base,
                  int T, int H, int E, int K, void* a_q, float* scale_a, int32_t* src2dst,
                  cudaStream_t st) {
  permute_quant_kernel<VPT, BLOCK><<<T, kQuantThreads, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), ids, bits, base, H, E, K,
      reinterpret_cast<uint8_t*>(a_q), scale_a, src2dst);
}

}  // namespace

// Scratch of moe_permute_quant_noalloc, for callers that cannot allocate:
// a fixed array in the library's device memory (held on every device that
// loads the library until exit) standing in for the caller's workspace.
// In host code the name is only a host-side handle, never a device address:
// permute_static_scratch() looks the device address up once per device.
static __device__ __align__(256) unsigned char g_permute_scratch[MOE_PERMUTE_NOALLOC_SCRATCH_BYTES];

void* permute_static_scratch() {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

size_t permute_ws_bytes(int T, int E) {
  const size_t C = (size_t)(T + 31) / 32;
  return 2 * align_up(C * (size_t)E * 4);
}

namespace {

template <bool BLOCK>
cudaError_t permute_quant(const void* x, const int32_t* ids, int T, int H, int E, int K,
                          void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets,
                          void* ws, int* err, cudaStream_t st) {
  const int C = (T + 31) / 32;
  uint32_t* bits = reinterpret_cast<uint32_t*>(ws);
  int32_t* base = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) +
                                             align_up((size_t)C * E * 4));
  if (C > 0) {
    const int blocks = (C + kBitsWarps - 1) / kBitsWarps;
    route_bits_kernel<<<blocks, kBitsWarps * 32, sizeof(uint32_t) * kBitsWarps * E, st>>>(
        ids, T, E, K, bits, err);
  }
  route_scan_kernel<<<1, 1024, 0, st>>>(bits, C, E, base, offsets);
  if (T > 0) {
    const int vpt = (H / 8 + kQuantThreads - 1) / kQuantThreads;
    if (vpt <= 1) launch_quant<1, BLOCK>(x, ids, bits, base, T, H, E, K, a_q, scale_a, src2dst, st);
    else if (vpt <= 2) launch_quant<2, BLOCK>(x, ids, bits, base, T, H, E, K, a_q, scale_a, src2dst, st);
    else if (vpt <= 4) launch_quant<4, BLOCK>(x, ids, bits, base, T, H, E, K, a_q, scale_a, src2dst, st);
    else if (vpt <= 8) launch_quant<8, BLOCK>(x, ids, bits, base, T, H, E, K, a_q, scale_a, src2dst, st);
    else launch_quant<16, BLOCK>(x, ids, bits, base, T, H, E, K, a_q, scale_a, src2dst, st);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_permute_quant(const void* x, const int32_t* ids, int T, int H, int E, int K,
                                 void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets,
                                 void* ws, int* err, cudaStream_t st) {
  return permute_quant<false>(x, ids, T, H, E, K, a_q, scale_a, src2dst, offsets, ws, err, st);
}

cudaError_t launch_permute_quant_block(const void* x, const int32_t* ids, int T, int H, int E,
                                       int K, void* a_q, float* scale_a, int32_t* src2dst,
                                       int32_t* offsets, void* ws, int* err, cudaStream_t st) {
  return permute_quant<true>(x, ids, T, H, E, K, a_q, scale_a, src2dst, offsets, ws, err, st);
}

}  // namespace moe
