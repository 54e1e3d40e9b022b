// moe_unpermute_sum: weighted post-reorder, out[t] = sum_k w[t,k] *
// down[src2dst[t*K+k]] accumulated in fp32 in slot order (the role of
// moe_sum_reduce in "[1/2] sgl-kernel: Fuse routed scaling factor into
// select_experts", sglang #8364, Motivation; routed_scaling_factor is
// already inside w). CTAs of 128 threads take one token and a slice of 1024
// columns, one 16-byte vector per thread (so small batches still spread over
// the SMs); 128-bit gathers of the K rows.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kVecPerBlock = 128;  // 16-byte vectors (1024 bf16) per CTA: one per thread

__global__ void __launch_bounds__(kThreads)
    unpermute_kernel(const __nv_bfloat16* __restrict__ down, const int32_t* __restrict__ src2dst,
                     const float* __restrict__ topk_w, int K, int H,
                     __nv_bfloat16* __restrict__ out, int* err) {
  chain_entry();
  __shared__ int64_t src[32];
  __shared__ float w[32];
  const int t = blockIdx.x;
  const int64_t M = (int64_t)gridDim.x * K;
  const int v0 = blockIdx.y * kVecPerBlock;
  if (threadIdx.x < K) {
    const int d = __ldg(src2dst + (int64_t)t * K + threadIdx.x);
    float wk = __ldg(topk_w + (int64_t)t * K + threadIdx.x);
    int64_t row = d;
    if (d < 0 || d >= M) {  // corrupt permutation: contribute nothing
      flag_error(err, MOE_DEV_BAD_EXPERT_ID);
      row = 0;
      wk = 0.0f;
    }
    src[threadIdx.x] = row * H;
    w[threadIdx.x] = wk;
  }
  __syncthreads();
  const int nvec = min(H >> 3, v0 + kVecPerBlock);
  uint4* o = reinterpret_cast<uint4*>(out + (int64_t)t * H);
  for (int i = v0 + threadIdx.x; i < nvec; i += kThreads) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k = 0; k < K; ++k) {
      float f[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(down + src[k]) + i), f);
      const float wk = w[k];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = __fmaf_rn(wk, f[j], acc[j]);
    }
    uint4 r;
    r.x = pack_bf16x2(acc[0], acc[1]);
    r.y = pack_bf16x2(acc[2], acc[3]);
    r.z = pack_bf16x2(acc[4], acc[5]);
    r.w = pack_bf16x2(acc[6], acc[7]);
    o[i] = r;
  }
}

}  // namespace

cudaError_t launch_unpermute_sum(const void* down, const int32_t* src2dst, const float* w,
                                 int T, int K, int H, void* out, int* err, cudaStream_t st,
                                 bool pdl) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(T, (H / 8 + kVecPerBlock - 1) / kVecPerBlock);
  return launch_kernel(unpermute_kernel, grid, dim3(kThreads), 0, st, pdl,
                       reinterpret_cast<const __nv_bfloat16*>(down), src2dst, w, K, H,
                       reinterpret_cast<__nv_bfloat16*>(out), err);
}

}  // namespace moe
