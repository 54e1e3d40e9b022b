// Device helpers shared by the kernels of the MoE layer forward (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_gb300.h"

namespace moe {

constexpr unsigned kFull = 0xffffffffu;

// Every kernel of the forward path starts with this: it waits for the kernel
// before it on the stream (when launched as its programmatic dependent), then
// lets the next one start its launch. A kernel therefore never runs ahead of
// the one before it, and when a kernel starts, every kernel two or more
// places earlier on the stream has completed.
__device__ __forceinline__ void chain_entry() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kern` on `st`. With `pdl` it is launched as a programmatic
// dependent of the previous kernel on the stream: its CTAs may be scheduled
// while that kernel still runs, and wait for it in chain_entry().
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// First fault wins; later ones are dropped.
__device__ __forceinline__ void flag_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// 8 bf16 packed in 16 bytes -> floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // .x = lo in the low half
  return *reinterpret_cast<uint32_t*>(&p);
}

// Two floats -> two e4m3 codes (round to nearest even, saturate to +-448),
// `a` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Per-token dynamic FP8 scale: max(amax, 1e-10) / 448 with IEEE division.
__device__ __forceinline__ float token_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
}

// 8 values x / scale (IEEE division) -> 8 e4m3 codes in 8 bytes.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float scale) {
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = e4m3x2(__fdiv_rn(f[2 * i], scale), __fdiv_rn(f[2 * i + 1], scale));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__device__ __forceinline__ float absmax8(const float (&f)[8], float m) {
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

}  // namespace moe
