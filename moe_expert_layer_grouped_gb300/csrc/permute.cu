// moe_permute_quant: pre-reorder with dynamic per-token FP8 quantisation
// ("Support token-level quantization for EP MoE", sglang #6782, Summary of
// Changes / Changelog / Code Review; expert row ranges from "Fix one bug in
// the grouped-gemm triton kernel", sglang #6772, Highlights).
//
// Batches with T <= 512 and T*K <= 4096 take one launch
// (permute_quant_small_kernel, below),
// larger ones three, all deterministic (no atomics whose order matters):
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
  chain_entry();
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
  chain_entry();
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

  // eight loads in flight per thread (the words are independent)
  int sum = 0;
  if (active) {
    int c = c0;
    for (; c + 8 <= c1; c += 8) {
      uint32_t w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = __ldg(bits + (int64_t)(c + u) * E + e);
#pragma unroll
      for (int u = 0; u < 8; ++u) sum += __popc(w[u]);
    }
    for (; c < c1; ++c) sum += __popc(__ldg(bits + (int64_t)c * E + e));
  }
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
    int c = c0;
    for (; c + 8 <= c1; c += 8) {
      uint32_t w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = __ldg(bits + (int64_t)(c + u) * E + e);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        base[(int64_t)(c + u) * E + e] = run;
        run += __popc(w[u]);
      }
    }
    for (; c < c1; ++c) {
      const int64_t i = (int64_t)c * E + e;
      base[i] = run;
      run += __popc(__ldg(bits + i));
    }
  }
}

constexpr int kQuantThreads = 128;

// Loads token t's row once (128-bit vectors, kept in registers), reduces its
// amax (per row, or per 128 channels when BLOCK), quantises it and stores the
// codes and scale to every destination row dst[0..K) >= 0. dst[] is written
// by threads 0..K-1 before the call; it is read only after a block barrier.
// With row_token (per-token scales only), the codes are stored once, in
// token order (row t of a_q, [T, H]), and row_token[d] = t is written for
// every destination row d instead; the scales still go to every d.
template <int VPT, bool BLOCK, int NT = kQuantThreads>
__device__ __forceinline__ void quant_scatter(const __nv_bfloat16* __restrict__ x, int t, int H,
                                              int K, const int* dst, float* red,
                                              uint8_t* __restrict__ a_q,
                                              float* __restrict__ scale_a,
                                              int32_t* __restrict__ row_token = nullptr) {
  const int tid = threadIdx.x;
  const int nvec = H >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)t * H);
  uint4 v[VPT];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = tid + i * NT;
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
      const int idx = tid + i * NT;
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
  for (int w = 1; w < NT / 32; ++w) amax = fmaxf(amax, red[w]);
  const float sc = token_scale(amax);
  if (tid < K && dst[tid] >= 0) {
    scale_a[dst[tid]] = sc;
    if (row_token != nullptr) row_token[dst[tid]] = t;
  }
  const Recip rb = recip_bracket(sc);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = tid + i * NT;
    if (idx < nvec) {
      float f[8];
      bf16x8_to_f32(v[i], f);
      const uint2 q = quant8(f, rb);
      if (row_token != nullptr) {
        *reinterpret_cast<uint2*>(a_q + (int64_t)t * H + (int64_t)idx * 8) = q;
        continue;
      }
      for (int k = 0; k < K; ++k) {
        const int d = dst[k];
        if (d >= 0) *reinterpret_cast<uint2*>(a_q + (int64_t)d * H + (int64_t)idx * 8) = q;
      }
    }
  }
}

// NVFP4: codes [T*K, H/2] (two E2M1 codes per byte, element 2j in the low
// nibble), one E4M3 scale per 16 channels sf [T*K, H/16], with the global
// scale g: scale code = e4m3((amax16 / 6) / g), codes = e2m1(x / (e4m3(code)
// * g)). A 16-channel block is two 8-value vectors, held by two adjacent
// threads (vector tid + i*NT, NT even), so its amax takes one shuffle. The
// token's vectors are all loaded before the first is used. When H % 256 == 0
// (whole warps of vectors: validity is warp-uniform) every eighth thread
// stores the scale bytes of four blocks as one word.
template <int VPT, int NT = kQuantThreads>
__device__ __forceinline__ void quant_scatter_nvfp4(const __nv_bfloat16* __restrict__ x, int t,
                                                    int H, int K, const int* dst, float g,
                                                    uint8_t* __restrict__ a_q,
                                                    uint8_t* __restrict__ sf) {
  static_assert(NT % 32 == 0, "whole warps");
  const int tid = threadIdx.x;
  const int nvec = H >> 3;
  const bool words = (H & 255) == 0;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)t * H);
  const Recip rg = recip_bracket(g);
  constexpr int G = VPT < 8 ? VPT : 8;  // vectors loaded ahead (16 spilled in the small kernel)
#pragma unroll
  for (int i0 = 0; i0 < VPT; i0 += G) {
    uint4 v[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int idx = tid + (i0 + j) * NT;
      if (idx < nvec) v[j] = __ldg(xr + idx);
    }
    if (i0 == 0) __syncthreads();  // dst[] is complete
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int i = i0 + j;
      const int idx = tid + i * NT;
      float f[8];
      float m = 0.0f;
      if (idx < nvec) {
        bf16x8_to_f32(v[j], f);
        m = absmax8(f, 0.0f);
      }
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
      uint32_t code = 0, q = 0;
      if (idx < nvec) {
        code = nvfp4_scale_code(m, g, rg);
        q = nvfp4_codes8(f, __fmul_rn(e4m3_value(code), g));
      }
      const uint32_t c2 = __shfl_down_sync(kFull, code, 2);
      const uint32_t c4 = __shfl_down_sync(kFull, code, 4);
      const uint32_t c6 = __shfl_down_sync(kFull, code, 6);
      if (idx < nvec) {
        const uint32_t word = code | (c2 << 8) | (c4 << 16) | (c6 << 24);
        for (int k = 0; k < K; ++k) {
          const int d = dst[k];
          if (d < 0) continue;
          *reinterpret_cast<uint32_t*>(a_q + (int64_t)d * (H >> 1) + (int64_t)idx * 4) = q;
          uint8_t* srow = sf + (int64_t)d * (H >> 4);
          if (words) {
            if ((idx & 7) == 0) *reinterpret_cast<uint32_t*>(srow + (idx >> 1)) = word;
          } else if ((idx & 1) == 0) {
            srow[idx >> 1] = (uint8_t)code;
          }
        }
      }
    }
  }
}

// BLOCK: one scale per 128 channels (scale_a [M, H/128]) instead of one per
// token. A 128-channel block is 16 vectors, held by the 16 lanes of a
// half-warp (vector tid + i*128 lies in block tid/16 + 8i), so its amax is a
// 16-lane shuffle reduction.
// QM: 0 per-token FP8, 1 block FP8, 2 NVFP4 (scale_a unused, sf / g used)
template <int VPT, int QM>  // VPT: 16-byte vectors (8 bf16) per thread
__global__ void __launch_bounds__(kQuantThreads)
    permute_quant_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ ids,
                         const uint32_t* __restrict__ bits, const int32_t* __restrict__ base,
                         int H, int E, int K, uint8_t* __restrict__ a_q,
                         float* __restrict__ scale_a, int32_t* __restrict__ src2dst,
                         int32_t* __restrict__ row_token, float g, uint8_t* __restrict__ sf) {
  chain_entry();
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
  if constexpr (QM == 2)
    quant_scatter_nvfp4<VPT>(x, t, H, K, dst, g, a_q, sf);
  else
    quant_scatter<VPT, QM == 1>(x, t, H, K, dst, red, a_q, scale_a, row_token);
}

// Small batches (T <= 512, T*K <= 4096): one launch does the routing and the
// quantisation. Every CTA (one per token) loads the whole batch's ids into
// shared memory, histograms them per expert and scans the histogram (the
// same offsets in every CTA; CTA 0 stores them), then ranks its own K slots
// among the earlier tokens' -- the stable counting sort of the three-launch
// path, with the same handling of bad ids: an id out of range gets
// destination -1, an id repeated within a token counts once and its repeats
// share the first one's row, and either raises MOE_DEV_BAD_EXPERT_ID.
constexpr int kSmallRoute = 4096;
constexpr int kSmallTokens = 512;  // every CTA re-reads all T*K ids: keep T small
#ifndef SMALL_THREADS
#define SMALL_THREADS 512
#endif
constexpr int kSmallThreads = SMALL_THREADS;  // more warps per token than the large path

template <int VPT, int QM>
__global__ void __launch_bounds__(kSmallThreads)
    permute_quant_small_kernel(const __nv_bfloat16* __restrict__ x,
                               const int32_t* __restrict__ ids, int T, int H, int E, int K,
                               uint8_t* __restrict__ a_q, float* __restrict__ scale_a,
                               int32_t* __restrict__ src2dst, int32_t* __restrict__ offsets,
                               int* err, int32_t* __restrict__ row_token, float g,
                               uint8_t* __restrict__ sf) {
  chain_entry();
  extern __shared__ int route_smem[];
  __shared__ int dst[32];
  __shared__ float red[kSmallThreads / 32];
  __shared__ int wpart[kSmallThreads / 32];
  const int n = T * K;
  int* raw = route_smem;    // [n] the ids as given
  int* s_ids = raw + n;     // [n] per slot: e (counts), E + e (a repeat of e), -1 (out of range)
  int* cnt = s_ids + n;     // [E]
  int* off = cnt + E;       // [E + 1]
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < n; i += kSmallThreads) raw[i] = __ldg(ids + i);
  for (int e = tid; e < E; e += kSmallThreads) cnt[e] = 0;
  __syncthreads();
  int bad = 0;
  for (int i = tid; i < n; i += kSmallThreads) {
    const int e = raw[i];
    int v = -1;
    if ((unsigned)e < (unsigned)E) {
      v = e;
      for (int j = i - i % K; j < i; ++j)
        if (raw[j] == e) v = E + e;
    }
    bad |= (v < 0 || v >= E);
    s_ids[i] = v;
  }
  bad = __syncthreads_or(bad);
  if (bad && t == 0 && tid == 0) flag_error(err, MOE_DEV_BAD_EXPERT_ID);
  for (int i = tid; i < n; i += kSmallThreads) {
    const int v = s_ids[i];
    if ((unsigned)v < (unsigned)E) atomicAdd(&cnt[v], 1);  // counts: order-free
  }
  __syncthreads();
  // exclusive scan of cnt over the block: ceil(E/128) consecutive experts per thread
  const int per = (E + kSmallThreads - 1) / kSmallThreads;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += cnt[e];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wpart[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += wpart[w];
  for (int e = e0; e < e1; ++e) {
    off[e] = run;
    run += cnt[e];
  }
  if (tid == kSmallThreads - 1) off[E] = run;
  __syncthreads();
  if (t == 0)
    for (int e = tid; e <= E; e += kSmallThreads) offsets[e] = off[e];
  // this token's slots: the rank of each of its experts among the earlier
  // tokens, by one pass over their slots with the token's experts marked in
  // a per-expert table (cnt[] is free again)
  const int prev = t * K;
  int* slot_of = cnt;
  __shared__ int rank[32];
  for (int e = tid; e < E; e += kSmallThreads) slot_of[e] = -1;
  if (tid < 32) rank[tid] = 0;
  __syncthreads();
  if (tid < K) {
    const int v = s_ids[prev + tid];
    if ((unsigned)v < (unsigned)E) slot_of[v] = tid;  // first occurrences are distinct
  }
  __syncthreads();
  for (int i = tid; i < prev; i += kSmallThreads) {
    const int v = s_ids[i];
    if ((unsigned)v < (unsigned)E) {
      const int k = slot_of[v];
      if (k >= 0) atomicAdd(&rank[k], 1);  // counts: order-free
    }
  }
  __syncthreads();
  if (tid < K) {
    const int v = s_ids[prev + tid];
    const int e = v >= E ? v - E : v;  // a repeat shares its expert's row
    const int d = v >= 0 ? off[e] + rank[slot_of[e]] : -1;
    dst[tid] = d;
    src2dst[(int64_t)t * K + tid] = d;
  }
  if constexpr (QM == 2)
    quant_scatter_nvfp4<VPT, kSmallThreads>(x, t, H, K, dst, g, a_q, sf);
  else
    quant_scatter<VPT, QM == 1, kSmallThreads>(x, t, H, K, dst, red, a_q, scale_a, row_token);
}

template <int VPT, int QM>
cudaError_t launch_small(const void* x, const int32_t* ids, int T, int H, int E, int K,
                         void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets, int* err,
                         cudaStream_t st, bool pdl, int32_t* row_token, float g, uint8_t* sf) {
  const size_t smem = sizeof(int) * (2 * (size_t)T * K + 2 * (size_t)E + 1);
  return launch_kernel(permute_quant_small_kernel<VPT, QM>, dim3(T), dim3(kSmallThreads),
                       smem, st, pdl, reinterpret_cast<const __nv_bfloat16*>(x), ids, T, H, E, K,
                       reinterpret_cast<uint8_t*>(a_q), scale_a, src2dst, offsets, err,
                       row_token, g, sf);
}

template <int VPT, int QM>
cudaError_t launch_quant(const void* x, const int32_t* ids, const uint32_t* bits,
                         const int32_t* base, int T, int H, int E, int K, void* a_q,
                         float* scale_a, int32_t* src2dst, cudaStream_t st, bool pdl,
                         int32_t* row_token, float g, uint8_t* sf) {
  return launch_kernel(permute_quant_kernel<VPT, QM>, dim3(T), dim3(kQuantThreads), 0, st,
                       pdl, reinterpret_cast<const __nv_bfloat16*>(x), ids, bits, base, H, E, K,
                       reinterpret_cast<uint8_t*>(a_q), scale_a, src2dst, row_token, g, sf);
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

template <int QM>
cudaError_t permute_quant(const void* x, const int32_t* ids, int T, int H, int E, int K,
                          void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets,
                          void* ws, int* err, cudaStream_t st, bool pdl,
                          int32_t* row_token = nullptr, float g = 0.0f, uint8_t* sf = nullptr) {
  if (T > 0 && T <= kSmallTokens && T * K <= kSmallRoute) {
    const int vpt = (H / 8 + kSmallThreads - 1) / kSmallThreads;
#define MOE_SMALL(V) launch_small<V, QM>(x, ids, T, H, E, K, a_q, scale_a, src2dst, offsets, err, st, pdl, row_token, g, sf)
    if (vpt <= 1) return MOE_SMALL(1);
    if (vpt <= 2) return MOE_SMALL(2);
    if (vpt <= 4) return MOE_SMALL(4);
    if (vpt <= 8) return MOE_SMALL(8);
    return MOE_SMALL(16);
#undef MOE_SMALL
  }
  const int C = (T + 31) / 32;
  uint32_t* bits = reinterpret_cast<uint32_t*>(ws);
  int32_t* base = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) +
                                             align_up((size_t)C * E * 4));
  cudaError_t e;
  if (C > 0) {
    const int blocks = (C + kBitsWarps - 1) / kBitsWarps;
    if ((e = launch_kernel(route_bits_kernel, dim3(blocks), dim3(kBitsWarps * 32),
                           sizeof(uint32_t) * kBitsWarps * E, st, pdl, ids, T, E, K, bits, err)))
      return e;
  }
  if ((e = launch_kernel(route_scan_kernel, dim3(1), dim3(1024), 0, st, pdl, bits, C, E, base,
                         offsets)))
    return e;
  if (T > 0) {
    const int vpt = (H / 8 + kQuantThreads - 1) / kQuantThreads;
#define MOE_QUANT(V) launch_quant<V, QM>(x, ids, bits, base, T, H, E, K, a_q, scale_a, src2dst, st, pdl, row_token, g, sf)
    if (vpt <= 1) return MOE_QUANT(1);
    if (vpt <= 2) return MOE_QUANT(2);
    if (vpt <= 4) return MOE_QUANT(4);
    if (vpt <= 8) return MOE_QUANT(8);
    return MOE_QUANT(16);
#undef MOE_QUANT
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_permute_quant(const void* x, const int32_t* ids, int T, int H, int E, int K,
                                 void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets,
                                 void* ws, int* err, cudaStream_t st, bool pdl,
                                 int32_t* row_token) {
  return permute_quant<0>(x, ids, T, H, E, K, a_q, scale_a, src2dst, offsets, ws, err, st, pdl,
                          row_token);
}

cudaError_t launch_permute_quant_block(const void* x, const int32_t* ids, int T, int H, int E,
                                       int K, void* a_q, float* scale_a, int32_t* src2dst,
                                       int32_t* offsets, void* ws, int* err, cudaStream_t st,
                                       bool pdl) {
  return permute_quant<1>(x, ids, T, H, E, K, a_q, scale_a, src2dst, offsets, ws, err, st, pdl);
}

cudaError_t launch_permute_quant_nvfp4(const void* x, const int32_t* ids, int T, int H, int E,
                                       int K, float g, void* a_q, uint8_t* sf, int32_t* src2dst,
                                       int32_t* offsets, void* ws, int* err, cudaStream_t st,
                                       bool pdl) {
  return permute_quant<2>(x, ids, T, H, E, K, a_q, nullptr, src2dst, offsets, ws, err, st, pdl,
                          nullptr, g, sf);
}

}  // namespace moe
