// moe_gate: grouped, bias-corrected top-k expert selection, one warp per
// token, with routed_scaling_factor fused into the renormalised weights
// ("[1/2] sgl-kernel: Fuse routed scaling factor into select_experts",
// sglang #8364, Motivation and Highlights).
//
// Lane l holds experts [l*EPL, (l+1)*EPL) in registers. Group scores (sum of
// the two largest biased scores per group) come from a butterfly merge of the
// lanes' top-2 pairs when a group is a power-of-two number of whole lanes
// (DeepSeek-V3: 4 lanes x 8 experts), else from a per-warp shared-memory copy
// of the keys. The topk_group groups and then the top_k experts are picked
// one at a time by two warp reductions (redux.sync): the largest
// order-preserving key, then the lowest index among the lanes holding it, so
// the result does not depend on scheduling and matches a sort with ties
// broken by the lower index.
//
// Every floating-point step that decides an id or a weight uses explicit
// round-to-nearest intrinsics (no contraction), so the fp32 scores are
// reproducible bit for bit by an independent implementation of the same
// operation sequence.
#include <float.h>
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// exp(x) in fp32: Cody-Waite reduction x = n*ln2 + r (ln2 split in a
// 16-significant-bit head and a tail), e^r by its degree-7 Taylor series
// (coefficients 1/k! rounded to fp32) in Horner form with fused
// multiply-adds, then two exact multiplications by powers of two.
__device__ __forceinline__ float exp32(float x) {
  if (x != x) return x;
  if (x > 88.8f) return CUDART_INF_F;
  if (x < -104.0f) return 0.0f;
  const float t = __fmul_rn(x, 0x1.715476p+0f);  // x * log2(e)
  const float n = rintf(t);
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, x);
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;            // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
  p = __fmaf_rn(p, r, 0.5f);             // 1/2!
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int ni = (int)n;
  const int n1 = ni / 2;
  const int n2 = ni - n1;
  const float y = __fmul_rn(p, __int_as_float((n1 + 127) << 23));
  return __fmul_rn(y, __int_as_float((n2 + 127) << 23));
}

// 1 / (1 + exp(-x)); the correctly rounded reciprocal is the correctly
// rounded quotient 1 / y, so this is the IEEE division's result
__device__ __forceinline__ float sigmoid32(float x) {
  return __frcp_rn(__fadd_rn(1.0f, exp32(-x)));
}

// Arg-max over the warp: larger value wins, equal values go to the lower
// index; `carry` travels with the winner. All lanes end with the winner.
__device__ __forceinline__ void warp_argmax(float& v, int& i, float& carry) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFull, v, o);
    const int oi = __shfl_xor_sync(kFull, i, o);
    const float oc = __shfl_xor_sync(kFull, carry, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
      carry = oc;
    }
  }
}

// Total order on fp32 keys as unsigned integers (larger float -> larger
// integer; -0 and +0 equal, as in IEEE comparison). 0 is below every key.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Of the lanes' candidates (key, index), the one with the largest key and,
// among equal keys, the lowest index (key 0: no candidate). Two warp
// reductions: the maximum key, then the minimum index among lanes holding it.
__device__ __forceinline__ int warp_pick(uint32_t key, uint32_t idx) {
  const uint32_t m = __reduce_max_sync(kFull, key);
  return (int)__reduce_min_sync(kFull, (key == m && key != 0u) ? idx : 0xFFFFFFFFu);
}

constexpr int kWarpsPerBlock = 4;

template <int EPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    gate_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E,
                int G, int TG, int K, int scoring, int renorm, float rsf,
                int32_t* __restrict__ ids_out, float* __restrict__ w_out, int n_shared) {
  chain_entry();
  extern __shared__ float keys_smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + warp;
  if (t >= T) return;  // warp-uniform
  const float* l = logits + (int64_t)t * E;
  const bool sigmoid = (scoring == MOE_SCORE_SIGMOID);

  float key[EPL], sv[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane * EPL + j;
    key[j] = -CUDART_INF_F;
    sv[j] = 0.0f;
    if (e < E) {
      const float lv = __ldg(l + e);
      if (sigmoid) {
        const float s = sigmoid32(lv);
        sv[j] = s;
        key[j] = bias ? __fadd_rn(s, __ldg(bias + e)) : s;
      } else {
        sv[j] = lv;
        key[j] = lv;
      }
    }
  }

  // ---- group-limited selection -------------------------------------------
  const int gsz = E / G;
  uint64_t kept = ~0ull;
  // groups made of whole lanes (a power-of-two number of them): the group's
  // two largest keys by a butterfly merge of per-lane top-2 pairs
  const int lpg = gsz / EPL;
  const bool lane_groups = TG < G && gsz % EPL == 0 && (lpg & (lpg - 1)) == 0;
  if (lane_groups) {
    float b1 = -CUDART_INF_F, b2 = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const float v = key[j];
      if (v > b1) {
        b2 = b1;
        b1 = v;
      } else if (v > b2) {
        b2 = v;
      }
    }
    for (int o = 1; o < lpg; o <<= 1) {
      const float ob1 = __shfl_xor_sync(kFull, b1, o);
      const float ob2 = __shfl_xor_sync(kFull, b2, o);
      const float n2 = fmaxf(fminf(b1, ob1), fmaxf(b2, ob2));
      b1 = fmaxf(b1, ob1);
      b2 = n2;
    }
    const float gscore = (gsz >= 2) ? __fadd_rn(b1, b2) : b1;
    const int gid = (lane * EPL) / gsz;
    const bool has = lane * EPL < E;
    const uint32_t gkey = has ? order_key(gscore) : 0u;
    kept = 0ull;
    for (int it = 0; it < TG; ++it)
      kept |= 1ull << warp_pick(((kept >> gid) & 1ull) ? 0u : gkey, (uint32_t)gid);
  } else if (TG < G) {
    // padded index e + e/32 keeps the group scans free of bank conflicts
    float* ks = keys_smem + warp * (E + (E >> 5) + 1);
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane * EPL + j;
      if (e < E) ks[e + (e >> 5)] = key[j];
    }
    __syncwarp();
    float gsc[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int g = lane + 32 * h;
      if (g < G) {
        float b1 = -CUDART_INF_F, b2 = -CUDART_INF_F;
        for (int i = 0; i < gsz; ++i) {
          const int e = g * gsz + i;
          const float v = ks[e + (e >> 5)];
          if (v > b1) {
            b2 = b1;
            b1 = v;
          } else if (v > b2) {
            b2 = v;
          }
        }
        gsc[h] = (gsz >= 2) ? __fadd_rn(b1, b2) : b1;
      }
    }
    kept = 0ull;
    uint32_t taken = 0;
    for (int it = 0; it < TG; ++it) {
      float bv = -CUDART_INF_F;
      int bi = 0x7fffffff;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int g = lane + 32 * h;
        if (g < G && !((taken >> h) & 1u) && (gsc[h] > bv || bi == 0x7fffffff)) {
          bv = gsc[h];
          bi = g;
        }
      }
      float dummy = 0.0f;
      warp_argmax(bv, bi, dummy);
      kept |= 1ull << bi;
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
  }

  // ---- top-k over the kept groups ----------------------------------------
  uint32_t open = 0;  // this lane's experts still eligible
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane * EPL + j;
    if (e < E && ((kept >> (e / gsz)) & 1ull)) open |= 1u << j;
  }
  uint32_t ok[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) ok[j] = order_key(key[j]);
  // this lane's best open expert (the first of equal keys: the lower index)
  uint32_t bk = 0u;
  int bj = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j)
    if (((open >> j) & 1u) && ok[j] > bk) {
      bk = ok[j];
      bj = j;
    }
  float my_s = 0.0f, S = 0.0f, m0 = 0.0f;
  int my_id = 0;
  for (int k = 0; k < K; ++k) {
    const int bi = warp_pick(bk, (uint32_t)(lane * EPL + bj));
    float sel = sv[0];
#pragma unroll
    for (int j = 1; j < EPL; ++j) sel = (bj == j) ? sv[j] : sel;
    const float bs = __shfl_sync(kFull, sel, bi / EPL);
    if (bi / EPL == lane) {  // the winner's lane takes its next best
      open &= ~(1u << bj);
      bk = 0u;
      bj = 0;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (((open >> j) & 1u) && ok[j] > bk) {
          bk = ok[j];
          bj = j;
        }
    }
    float term = bs;
    if (!sigmoid) {
      if (k == 0) m0 = bs;
      term = exp32(__fsub_rn(bs, m0));
    }
    if (lane == k) {
      my_s = term;
      my_id = bi;
    }
    S = __fadd_rn(S, term);
  }

  float wk;
  if (sigmoid) {
    wk = renorm ? __fmul_rn(__fdiv_rn(my_s, S), rsf) : __fmul_rn(my_s, rsf);
  } else if (renorm) {
    wk = __fmul_rn(__fdiv_rn(my_s, S), rsf);
  } else {
    // full softmax probability of the selected expert: max over all logits,
    // denominator summed over experts in index order
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (lane * EPL + j < E) mx = fmaxf(mx, sv[j]);
    mx = warp_max(mx);
    float Z = 0.0f;
    if (lane == 0)
      for (int e = 0; e < E; ++e) Z = __fadd_rn(Z, exp32(__fsub_rn(__ldg(l + e), mx)));
    Z = __shfl_sync(kFull, Z, 0);
    // my_s holds exp(l_k - l_slot0); recompute against the global max
    float lk = 0.0f;
    // the selected logit: slot k's logit = l[my_id]
    if (lane < K) lk = __ldg(l + my_id);
    wk = __fmul_rn(__fdiv_rn(exp32(__fsub_rn(lk, mx)), Z), rsf);
  }
  // rows of K + n_shared slots: the routed picks, then the shared experts
  // (ids E .. E+n_shared-1, weight 1)
  const int64_t row = (int64_t)t * (K + n_shared);
  if (lane < K) {
    ids_out[row + lane] = my_id;
    w_out[row + lane] = wk;
  } else if (lane < K + n_shared) {
    ids_out[row + lane] = E + (lane - K);
    w_out[row + lane] = 1.0f;
  }
}

template <int EPL>
cudaError_t launch_epl(const float* logits, const float* bias, int T, int E, int G, int TG,
                       int K, int scoring, int renorm, float rsf, int32_t* ids, float* w,
                       int S, cudaStream_t st) {
  const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const size_t smem = (TG < G) ? sizeof(float) * kWarpsPerBlock * (E + (E >> 5) + 1) : 0;
  gate_kernel<EPL><<<blocks, kWarpsPerBlock * 32, smem, st>>>(logits, bias, T, E, G, TG, K,
                                                              scoring, renorm, rsf, ids, w, S);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate(const float* logits, const float* bias, int T, int E, int G, int TG,
                        int K, int scoring, int renorm, float rsf, int32_t* ids, float* w,
                        int n_shared, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int S = n_shared;
  const int per_lane = (E + 31) / 32;
  if (per_lane <= 1) return launch_epl<1>(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st);
  if (per_lane <= 2) return launch_epl<2>(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st);
  if (per_lane <= 4) return launch_epl<4>(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st);
  if (per_lane <= 8) return launch_epl<8>(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st);
  if (per_lane <= 16) return launch_epl<16>(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st);
  return launch_epl<32>(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st);
}

}  // namespace moe
