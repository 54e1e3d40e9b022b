// Device helpers shared by the kernels of the MoE layer forward (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp4.h>
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

// ---- quotients rounded to a narrow format -----------------------------------
// A quantiser's code is narrow(fl(x / d)): the fp32 quotient (IEEE division,
// nearest even), then rounded to e4m3 or e2m1 (nearest even, saturating).
// The division is avoided where it cannot change the code. With r = rcp_rn(d)
// a normal number, rl = fl(r (1 - 2^-20)) and rh = fl(r (1 + 2^-20)), the
// exact products x*rl and x*rh lie within a relative 3 * 2^-24 of
// x (1 -+ 2^-20) / d, so below and above fl(x / d), which is within 2^-24 of
// x / d; rounding them to fp32 keeps that order (rounding is monotone). Since
// the narrow rounding is monotone as well, where fl(x*rl) and fl(x*rh) give
// the same code, fl(x / d) gives it too. The IEEE quotient is computed only
// for the rare x / d within ~2^-20 of a rounding boundary of the narrow
// format (and when r is outside [2^-125, 2^126], where the bounds above do
// not hold or the products could meet inf * 0).
struct Recip {
  float d, lo, hi;
  bool ok;
};

__device__ __forceinline__ Recip recip_bracket(float d) {
  const float r = __frcp_rn(d);
  Recip b;
  b.d = d;
  b.lo = __fmul_rn(r, 1.0f - 0x1p-20f);
  b.hi = __fmul_rn(r, 1.0f + 0x1p-20f);
  b.ok = r >= 0x1p-125f && r <= 0x1p126f;
  return b;
}

// 8 values x / d -> 8 e4m3 codes in 8 bytes (x / d as above).
__device__ __forceinline__ uint2 quant8(const float (&f)[8], const Recip& b) {
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo[i] = e4m3x2(__fmul_rn(f[2 * i], b.lo), __fmul_rn(f[2 * i + 1], b.lo));
    hi[i] = e4m3x2(__fmul_rn(f[2 * i], b.hi), __fmul_rn(f[2 * i + 1], b.hi));
  }
  uint2 q = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
  const uint2 qh = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
  if (!b.ok || q.x != qh.x || q.y != qh.y) {
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = e4m3x2(__fdiv_rn(f[2 * i], b.d), __fdiv_rn(f[2 * i + 1], b.d));
    q = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
  return q;
}

__device__ __forceinline__ uint2 quant8(const float (&f)[8], float scale) {
  return quant8(f, recip_bracket(scale));
}

__device__ __forceinline__ float absmax8(const float (&f)[8], float m) {
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// ---- NVFP4 (E2M1 elements, one E4M3 scale per 16 along K, fp32 global
// scale g) ------------------------------------------------------------------

// Exact value of an e4m3 code (every e4m3 value is an fp16 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// Block scale of 16 values with largest magnitude amax: the e4m3 code of
// (amax / 6) / g (IEEE divisions, round to nearest even, saturating). The
// brackets of the quotients above, applied twice: fl(amax * 6l) <= fl(amax
// / 6) <= fl(amax * 6h), and each bound times gl / gh (monotone again) stays
// on its side of fl(fl(amax / 6) / g). rg is the Recip of g.
__device__ __forceinline__ uint32_t nvfp4_scale_code(float amax, float g, const Recip& rg) {
  const float r6 = 1.0f / 6.0f;  // rcp_rn(6), a normal number
  const float lo = __fmul_rn(__fmul_rn(amax, __fmul_rn(r6, 1.0f - 0x1p-20f)), rg.lo);
  const float hi = __fmul_rn(__fmul_rn(amax, __fmul_rn(r6, 1.0f + 0x1p-20f)), rg.hi);
  const uint32_t c = e4m3x2(lo, hi);
  if (rg.ok && (c & 0xFFu) == (c >> 8)) return c & 0xFFu;
  return e4m3x2(__fdiv_rn(__fdiv_rn(amax, 6.0f), g), 0.0f) & 0xFFu;
}

__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
}

// 8 values -> 8 E2M1 codes x / step (IEEE division, nearest even,
// saturating to +-6; the quotient brackets above), element 2j in the low
// nibble of byte j; all zero when step is 0.
__device__ __forceinline__ uint32_t nvfp4_codes8(const float (&f)[8], float step) {
  if (!(step > 0.0f)) return 0u;
  const Recip b = recip_bracket(step);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    lo |= e2m1x2(__fmul_rn(f[2 * j], b.lo), __fmul_rn(f[2 * j + 1], b.lo)) << (8 * j);
    hi |= e2m1x2(__fmul_rn(f[2 * j], b.hi), __fmul_rn(f[2 * j + 1], b.hi)) << (8 * j);
  }
  if (b.ok && lo == hi) return lo;
  uint32_t r = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    r |= e2m1x2(__fdiv_rn(f[2 * j], step), __fdiv_rn(f[2 * j + 1], step)) << (8 * j);
  return r;
}

}  // namespace moe
