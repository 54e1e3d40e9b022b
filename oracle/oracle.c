/*
 * Oracle for the grouped-expert MoE layer forward: plain, slow, CPU-only C.
 *
 * TEST INFRASTRUCTURE, not part of the product: only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it. It shares no code
 * with the CUDA library. Build with:  gcc -O2 -std=c11 -ffp-contract=off
 * -fopenmp -fPIC -shared oracle.c -lm   (no fast-math: the fp32 steps below
 * rely on IEEE single-precision semantics, one rounding per operation).
 *
 * Citations name the page and section they come from:
 *   [P1] "Fix one bug in the grouped-gemm triton kernel" (sglang #6772)
 *   [P2] "Support token-level quantization for EP MoE" (sglang #6782)
 *   [P3] "[1/2] sgl-kernel: Fuse routed scaling factor into select_experts"
 *        (sglang #8364)
 *
 * Parity pins: every function here is pinned by a CPU test against a value
 * or property fixed by the pages or by mathematics (hand-worked gate cases,
 * brute-force top-k enumeration, sum-of-weights invariant, permutation
 * bijection and identity, exhaustive FP8 nearest-value search, exact-integer
 * and dense-matmul special cases of the GEMM, a dense MLP for E=1,K=1; for
 * NVFP4 the format's magnitude list, an exhaustive E2M1 nearest-even search,
 * the quantiser in closed form and exact power-of-two-scaled GEMMs).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* threads                                                             */
/* ------------------------------------------------------------------ */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* fp32 exponential and logistic function                             */
/*                                                                     */
/* The pages do not say how exp is evaluated. The gate's top-k ids are */
/* decided on fp32 sigmoid scores, so the oracle and the kernel must   */
/* produce the same fp32 score. Both evaluate exp with the same        */
/* published method, each written independently:                      */
/*   Cody & Waite argument reduction x = n*ln2 + r, |r| <= ln2/2, with */
/*   ln2 split into a 16-bit-mantissa high part and a low correction;  */
/*   e^r by its Taylor series to degree 7 (coefficients 1/k! rounded   */
/*   to fp32) in Horner form with fused multiply-adds; then scaling by */
/*   2^n in two exact power-of-two multiplications.                     */
/* ------------------------------------------------------------------ */
static float pow2_int(int k) { /* 2^k for k in [-126, 127] */
  uint32_t b = (uint32_t)(k + 127) << 23;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

float oracle_exp32(float x) {
  if (x != x) return x;
  if (x > 88.8f) return INFINITY;
  if (x < -104.0f) return 0.0f;
  const float log2e = 0x1.715476p+0f;
  const float ln2_hi = 0x1.62e4p-1f;
  const float ln2_lo = 0x1.7f7d1cp-20f;
  float t = x * log2e;
  float n = rintf(t);
  float r = fmaf(-n, ln2_hi, x);
  r = fmaf(-n, ln2_lo, r);
  float p = 0x1.a01a02p-13f;        /* 1/7! */
  p = fmaf(p, r, 0x1.6c16c2p-10f);  /* 1/6! */
  p = fmaf(p, r, 0x1.111112p-7f);   /* 1/5! */
  p = fmaf(p, r, 0x1.555556p-5f);   /* 1/4! */
  p = fmaf(p, r, 0x1.555556p-3f);   /* 1/3! */
  p = fmaf(p, r, 0.5f);             /* 1/2! */
  p = fmaf(p, r, 1.0f);             /* 1/1! */
  p = fmaf(p, r, 1.0f);             /* 1/0! */
  int ni = (int)n;
  int n1 = ni / 2;
  int n2 = ni - n1;
  float y = p * pow2_int(n1);
  return y * pow2_int(n2);
}

void oracle_exp32_n(const float* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_exp32(x[i]);
}

float oracle_sigmoid32(float x) {
  float e = oracle_exp32(-x);
  float d = 1.0f + e;
  return 1.0f / d;
}

void oracle_sigmoid32_n(const float* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_sigmoid32(x[i]);
}

/* ------------------------------------------------------------------ */
/* FP8 e4m3 ("fn" variant: no infinities, 0x7F/0xFF are NaN)           */
/* [P2] names FP8 activations without fixing the format; the reading   */
/* is OCP e4m3: exponent bias 7, 3 mantissa bits, largest finite 448,  */
/* subnormals m * 2^-9. Encoding rounds to nearest, ties to the even   */
/* mantissa, and saturates to +-448 instead of producing NaN; the sign */
/* of zero is kept.                                                    */
/* ------------------------------------------------------------------ */
uint8_t oracle_e4m3_encode(float x) {
  uint32_t bits;
  memcpy(&bits, &x, 4);
  uint8_t sign = (bits >> 31) ? 0x80 : 0x00;
  if (x != x) return (uint8_t)(sign | 0x7F);
  float a = fabsf(x);
  if (a >= 448.0f) return (uint8_t)(sign | 0x7E);
  if (a < 0x1p-6f) {
    /* subnormal range: units of 2^-9, value m * 2^-9, m in 0..8 */
    float u = a * 0x1p9f; /* exact: power-of-two scaling */
    int m = (int)rintf(u);
    /* m == 8 is the smallest normal, code 0x08: same bit pattern */
    return (uint8_t)(sign | m);
  }
  int ex;
  frexpf(a, &ex); /* a = f * 2^ex, f in [0.5, 1) -> a in [2^(ex-1), 2^ex) */
  int E = ex - 1; /* unbiased exponent, a in [2^E, 2^(E+1)) */
  /* units of the e4m3 ulp 2^(E-3): u in [8, 16), exact */
  float u = ldexpf(a, 3 - E);
  int m = (int)rintf(u);
  if (m == 16) {
    m = 8;
    E += 1;
  }
  int be = E + 7;
  int code = (be << 3) | (m - 8);
  if (code > 0x7E) code = 0x7E; /* saturate (0x7F would be NaN) */
  return (uint8_t)(sign | code);
}

void oracle_e4m3_encode_n(const float* x, uint8_t* q, int64_t n) {
  for (int64_t i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(x[i]);
}

double oracle_e4m3_decode(uint8_t q) {
  int s = q >> 7;
  int e = (q >> 3) & 15;
  int m = q & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

static double g_e4m3_lut[256];
static int g_lut_ready = 0;
static void init_lut(void) {
  if (g_lut_ready) return;
  for (int i = 0; i < 256; ++i) g_e4m3_lut[i] = oracle_e4m3_decode((uint8_t)i);
  g_lut_ready = 1;
}

/* ------------------------------------------------------------------ */
/* bf16                                                                */
/* ------------------------------------------------------------------ */
static float bf16_to_f32(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

uint16_t oracle_bf16_round(double v) {
  /* round to odd into fp32 first, so the final round to nearest even into
   * bf16 is a single correct rounding of v */
  float f = (float)v;
  if (v == v && !isinf(f) && (double)f != v) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if (fabs((double)f) > fabs(v)) b -= 1;
    b |= 1u;
    memcpy(&f, &b, 4);
  }
  uint32_t b;
  memcpy(&b, &f, 4);
  if (f != f) return 0x7FC0;
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

void oracle_bf16_round_n(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(v[i]);
}

/* ------------------------------------------------------------------ */
/* Gate                                                                */
/*                                                                     */
/* [P3] Motivation/Highlights: the gate normalises the selected top-k  */
/* weights and multiplies them by routed_scaling_factor. [P3] names    */
/* the grouped, bias-corrected selection (biased_grouped_topk). The    */
/* pages do not spell out the arithmetic; the readings taken here:     */
/*  - sigmoid scoring: s = 1/(1+exp(-l)) in fp32; the selection key is */
/*    b = s + bias (fp32); a group's score is the sum of its two       */
/*    largest keys (its only key when groups hold one expert);         */
/*  - the topk_group best groups are kept, then the top_k best keys    */
/*    among the kept groups' experts; ties go to the lower index, both */
/*    for groups and experts; slot k holds the k-th selection;         */
/*  - weights use the unbiased s: w_k = (s_k / S) * rsf with S the     */
/*    fp32 sum of the selected s in slot order (renormalise), or       */
/*    w_k = s_k * rsf without renormalisation;                         */
/*  - softmax scoring (one group, no bias): experts are selected by     */
/*    logit, which orders exactly like softmax; with renormalisation   */
/*    w_k = (exp(l_k - l_0) / S) * rsf, S the slot-order fp32 sum of   */
/*    those exponentials; without it the denominator is the sum over   */
/*    all experts in index order with l_max subtracted.                */
/* ------------------------------------------------------------------ */
typedef struct {
  float key;
  int idx;
} kv_t;

static int cmp_kv_desc(const void* pa, const void* pb) {
  const kv_t* a = (const kv_t*)pa;
  const kv_t* b = (const kv_t*)pb;
  if (a->key > b->key) return -1;
  if (a->key < b->key) return 1;
  return (a->idx < b->idx) ? -1 : (a->idx > b->idx ? 1 : 0);
}

static int gate_check(int T, int E, int G, int TG, int K, int scoring,
                      const float* bias) {
  if (T < 0 || E < 1 || G < 1 || E % G != 0) return -1;
  if (TG < 1 || TG > G) return -1;
  if (K < 1 || K > TG * (E / G)) return -1;
  if (scoring != ORACLE_SIGMOID && scoring != ORACLE_SOFTMAX) return -1;
  if (scoring == ORACLE_SOFTMAX && (bias != NULL || G != 1)) return -2;
  return 0;
}

/* one token; scratch holds 2*E kv_t + E floats */
static void gate_token(const float* l, const float* bias, int E, int G, int TG,
                       int K, int scoring, int renorm, float rsf, int32_t* ids,
                       float* w, kv_t* kv, kv_t* gkv, float* s) {
  const int gsz = E / G;
  for (int e = 0; e < E; ++e) {
    if (scoring == ORACLE_SIGMOID) {
      s[e] = oracle_sigmoid32(l[e]);
      kv[e].key = bias ? s[e] + bias[e] : s[e];
    } else {
      s[e] = l[e];
      kv[e].key = l[e];
    }
    kv[e].idx = e;
  }
  /* group scores */
  int allowed_all = (TG == G);
  unsigned char* allowed = (unsigned char*)calloc((size_t)G, 1);
  if (!allowed_all) {
    for (int g = 0; g < G; ++g) {
      float b1 = -INFINITY, b2 = -INFINITY;
      for (int j = 0; j < gsz; ++j) {
        float v = kv[g * gsz + j].key;
        if (v > b1) {
          b2 = b1;
          b1 = v;
        } else if (v > b2) {
          b2 = v;
        }
      }
      gkv[g].key = (gsz >= 2) ? (b1 + b2) : b1;
      gkv[g].idx = g;
    }
    qsort(gkv, (size_t)G, sizeof(kv_t), cmp_kv_desc);
    for (int i = 0; i < TG; ++i) allowed[gkv[i].idx] = 1;
  }
  /* candidates of the kept groups, sorted by key */
  int nc = 0;
  kv_t* cand = gkv + G; /* scratch after the group entries */
  for (int e = 0; e < E; ++e) {
    if (allowed_all || allowed[e / gsz]) cand[nc++] = kv[e];
  }
  free(allowed);
  qsort(cand, (size_t)nc, sizeof(kv_t), cmp_kv_desc);
  for (int k = 0; k < K; ++k) ids[k] = cand[k].idx;

  if (scoring == ORACLE_SIGMOID) {
    if (renorm) {
      float S = 0.0f;
      for (int k = 0; k < K; ++k) S = S + s[ids[k]];
      for (int k = 0; k < K; ++k) w[k] = (s[ids[k]] / S) * rsf;
    } else {
      for (int k = 0; k < K; ++k) w[k] = s[ids[k]] * rsf;
    }
  } else {
    if (renorm) {
      float m = l[ids[0]];
      float S = 0.0f;
      for (int k = 0; k < K; ++k) S = S + oracle_exp32(l[ids[k]] - m);
      for (int k = 0; k < K; ++k) w[k] = (oracle_exp32(l[ids[k]] - m) / S) * rsf;
    } else {
      float m = l[0];
      for (int e = 1; e < E; ++e)
        if (l[e] > m) m = l[e];
      float Z = 0.0f;
      for (int e = 0; e < E; ++e) Z = Z + oracle_exp32(l[e] - m);
      for (int k = 0; k < K; ++k) w[k] = (oracle_exp32(l[ids[k]] - m) / Z) * rsf;
    }
  }
}

int oracle_gate(const float* logits, const float* bias, int T, int E,
                int num_groups, int topk_group, int top_k, int scoring,
                int renormalize, float routed_scaling_factor,
                int32_t* topk_ids, float* topk_w) {
  int rc = gate_check(T, E, num_groups, topk_group, top_k, scoring, bias);
  if (rc) return rc;
#pragma omp parallel
  {
    kv_t* kv = (kv_t*)malloc(sizeof(kv_t) * (size_t)E);
    kv_t* gkv = (kv_t*)malloc(sizeof(kv_t) * (size_t)(E + num_groups));
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      gate_token(logits + (int64_t)t * E, bias, E, num_groups, topk_group, top_k,
                 scoring, renormalize, routed_scaling_factor,
                 topk_ids + (int64_t)t * top_k, topk_w + (int64_t)t * top_k, kv,
                 gkv, s);
    }
    free(kv);
    free(gkv);
    free(s);
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Routing / pre-reorder                                               */
/* [P2] Code Review: the per-token scales are written in permuted      */
/* order through src2dst after the pre-reorder. [P1] Highlights: each  */
/* expert owns a contiguous row range starting at m_range_start.       */
/* Reading: a counting sort of the flattened index i = t*K + k by      */
/* expert, stable in i, so an expert's rows hold its tokens in         */
/* ascending token order; offsets[0] = 0, offsets[e+1] = offsets[e] +  */
/* count[e]; empty experts own an empty range.                         */
/* ------------------------------------------------------------------ */
void oracle_route(const int32_t* topk_ids, int T, int E, int K,
                  int32_t* offsets, int32_t* src2dst) {
  int64_t n = (int64_t)T * K;
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (int64_t i = 0; i < n; ++i) offsets[topk_ids[i] + 1] += 1;
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  for (int64_t i = 0; i < n; ++i) {
    int e = topk_ids[i];
    src2dst[i] = offsets[e] + fill[e];
    fill[e] += 1;
  }
  free(fill);
}

/* [P2] Summary/Changelog: per-token maximum values give the per-token
 * dynamic FP8 scales. Reading: amax = max |x| over the row's bf16 values,
 * scale = max(amax, 1e-10) / 448 in fp32, code = e4m3(x / scale) with an
 * IEEE fp32 division; dequantised value = code * scale. */
void oracle_row_quant(const uint16_t* x, int64_t R, int C, uint8_t* q,
                      float* scale) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    const uint16_t* row = x + r * C;
    float amax = 0.0f;
    for (int c = 0; c < C; ++c) {
      float v = fabsf(bf16_to_f32(row[c]));
      if (v > amax) amax = v;
    }
    float sc = fmaxf(amax, 1e-10f) / 448.0f;
    scale[r] = sc;
    for (int c = 0; c < C; ++c) q[r * C + c] = oracle_e4m3_encode(bf16_to_f32(row[c]) / sc);
  }
}

void oracle_permute_quant(const uint16_t* x, const int32_t* topk_ids, int T,
                          int H, int E, int K, uint8_t* a_q, float* scale_a,
                          int32_t* src2dst, int32_t* offsets) {
  oracle_route(topk_ids, T, E, K, offsets, src2dst);
  uint8_t* q = (uint8_t*)malloc((size_t)T * H);
  float* sc = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
  oracle_row_quant(x, T, H, q, sc);
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      int64_t d = src2dst[(int64_t)t * K + k];
      memcpy(a_q + d * H, q + (int64_t)t * H, (size_t)H);
      scale_a[d] = sc[t];
    }
  }
  free(q);
  free(sc);
}

/* ------------------------------------------------------------------ */
/* Grouped GEMM                                                        */
/* [P1] Highlights and [P2] Changelog: per expert, over its row range, */
/* the accumulator is dequantised by scale_a of the ROW (per token)    */
/* times the weight scale; no block quantisation. Reading: the weight  */
/* scale is per output channel, scale_b[e,n]. The dot product is taken */
/* over exactly decoded FP8 values in fp64: every product is exact and */
/* for K <= 2^13 the sum is exact as well (products lie in            */
/* [2^-18, 2^18], so partial sums need at most 36 + 13 < 53 bits).     */
/* ------------------------------------------------------------------ */
void oracle_grouped_gemm(const uint8_t* A, const float* scale_a,
                         const uint8_t* B, const float* scale_b,
                         const int32_t* offsets, int M, int N, int Kd, int E,
                         double* C) {
  init_lut();
  int32_t* row_e = (int32_t*)malloc(sizeof(int32_t) * (size_t)(M > 0 ? M : 1));
  for (int r = 0; r < M; ++r) row_e[r] = -1;
  for (int e = 0; e < E; ++e)
    for (int r = offsets[e]; r < offsets[e + 1] && r < M; ++r) row_e[r] = e;
#pragma omp parallel
  {
    double* a = (double*)malloc(sizeof(double) * (size_t)Kd);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < M; ++r) {
      int e = row_e[r];
      double* c = C + (int64_t)r * N;
      if (e < 0) {
        for (int n = 0; n < N; ++n) c[n] = 0.0;
        continue;
      }
      for (int k = 0; k < Kd; ++k) a[k] = g_e4m3_lut[A[(int64_t)r * Kd + k]];
      const uint8_t* Be = B + (int64_t)e * N * Kd;
      for (int n = 0; n < N; ++n) {
        const uint8_t* b = Be + (int64_t)n * Kd;
        double acc = 0.0;
        for (int k = 0; k < Kd; ++k) acc += a[k] * g_e4m3_lut[b[k]];
        c[n] = acc * (double)scale_a[r] * (double)scale_b[(int64_t)e * N + n];
      }
    }
    free(a);
  }
  free(row_e);
}

/* [P2] Code Review: the activation between the GEMMs produces
 * down_input. Reading: the first I output channels of w13 are the gate
 * projection g, the next I the up projection u; h = silu(g) * u with
 * silu(g) = g / (1 + exp(-g)), in fp64. */
void oracle_silu_mul(const double* C, int64_t M, int I, double* h) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < M; ++r) {
    for (int j = 0; j < I; ++j) {
      double g = C[r * 2 * I + j];
      double u = C[r * 2 * I + I + j];
      h[r * I + j] = g / (1.0 + exp(-g)) * u;
    }
  }
}

/* Post-reorder: weighted sum of each token's K expert outputs, fp64. */
void oracle_unpermute_sum(const double* down, const int32_t* src2dst,
                          const float* topk_w, int T, int K, int H,
                          double* out) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double* o = out + (int64_t)t * H;
    for (int c = 0; c < H; ++c) o[c] = 0.0;
    for (int k = 0; k < K; ++k) {
      double w = (double)topk_w[(int64_t)t * K + k];
      const double* d = down + (int64_t)src2dst[(int64_t)t * K + k] * H;
      for (int c = 0; c < H; ++c) o[c] += w * d[c];
    }
  }
}

/* ------------------------------------------------------------------ */
/* Whole layer, token by token                                         */
/* The layer's steps in the pages' order: gate [P3], pre-reorder with  */
/* per-token FP8 [P2], w13 GEMM with per-row scale_a [P1][P2], SiLU*mul */
/* and per-token requantisation [P2], w2 GEMM, weighted post-reorder.  */
/* A token's output depends on that token alone, so the permutation   */
/* reduces to visiting the token's K experts; h is rounded to bf16,    */
/* the activation dtype, before its per-token requantisation.          */
/* ------------------------------------------------------------------ */
int oracle_forward_tokens(const uint16_t* x, const float* logits,
                          const float* bias, const uint8_t* w13,
                          const float* s13, const uint8_t* w2, const float* s2,
                          int T, int H, int I, int E, int num_groups,
                          int topk_group, int top_k, int scoring,
                          int renormalize, float routed_scaling_factor,
                          const int64_t* tokens, int n_tok, double* out,
                          int32_t* ids_out, float* w_out) {
  return oracle_forward_tokens_shared(x, logits, bias, w13, s13, w2, s2, T, H, I, E, 0,
                                      num_groups, topk_group, top_k, scoring, renormalize,
                                      routed_scaling_factor, tokens, n_tok, out, ids_out,
                                      w_out);
}

/* The layer with n_shared shared experts ("[1/2] sgl-kernel: Fuse routed
 * scaling factor into select_experts", sglang #8364, Highlights: shared expert
 * fusion alongside the fused scaling factor). Reading: every token also runs
 * experts E .. E+n_shared-1 of w13/w2, each added with weight 1 after the K
 * routed slots (routed_scaling_factor is already inside the routed weights),
 * i.e. the DeepSeek-V3 layer output shared(x) + sum_k w_k expert_k(x). */
int oracle_forward_tokens_shared(const uint16_t* x, const float* logits,
                                 const float* bias, const uint8_t* w13,
                                 const float* s13, const uint8_t* w2, const float* s2,
                                 int T, int H, int I, int E, int n_shared,
                                 int num_groups, int topk_group, int top_k, int scoring,
                                 int renormalize, float routed_scaling_factor,
                                 const int64_t* tokens, int n_tok, double* out,
                                 int32_t* ids_out, float* w_out) {
  int rc = gate_check(T, E, num_groups, topk_group, top_k, scoring, bias);
  if (rc) return rc;
  if (n_shared < 0) return -1;
  for (int i = 0; i < n_tok; ++i)
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
  init_lut();
  const int K = top_k;
  const int N13 = 2 * I;
  int status = 0;
#pragma omp parallel
  {
    kv_t* kv = (kv_t*)malloc(sizeof(kv_t) * (size_t)E);
    kv_t* gkv = (kv_t*)malloc(sizeof(kv_t) * (size_t)(E + num_groups));
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    double* c = (double*)malloc(sizeof(double) * (size_t)N13);
    uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    double* h2 = (double*)malloc(sizeof(double) * (size_t)I);
    int32_t ids[64];
    float w[64];
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < n_tok; ++i) {
      int64_t t = tokens[i];
      double* o = out + (int64_t)i * H;
      if (K > 64) {
        status = -2;
        continue;
      }
      gate_token(logits + t * E, bias, E, num_groups, topk_group, K, scoring,
                 renormalize, routed_scaling_factor, ids, w, kv, gkv, s);
      if (ids_out)
        for (int k = 0; k < K; ++k) ids_out[(int64_t)i * K + k] = ids[k];
      if (w_out)
        for (int k = 0; k < K; ++k) w_out[(int64_t)i * K + k] = w[k];
      /* per-token quantisation of the hidden state */
      const uint16_t* xr = x + t * H;
      float amax = 0.0f;
      for (int hh = 0; hh < H; ++hh) {
        float v = fabsf(bf16_to_f32(xr[hh]));
        if (v > amax) amax = v;
      }
      float sa = fmaxf(amax, 1e-10f) / 448.0f;
      for (int hh = 0; hh < H; ++hh)
        a[hh] = g_e4m3_lut[oracle_e4m3_encode(bf16_to_f32(xr[hh]) / sa)];
      for (int cc = 0; cc < H; ++cc) o[cc] = 0.0;
      for (int k = 0; k < K + n_shared; ++k) {
        /* routed slots, then the shared experts with weight 1 */
        const int e = k < K ? ids[k] : E + (k - K);
        const uint8_t* We = w13 + (int64_t)e * N13 * H;
        for (int n = 0; n < N13; ++n) {
          const uint8_t* b = We + (int64_t)n * H;
          double acc = 0.0;
          for (int hh = 0; hh < H; ++hh) acc += a[hh] * g_e4m3_lut[b[hh]];
          c[n] = acc * (double)sa * (double)s13[(int64_t)e * N13 + n];
        }
        float amax2 = 0.0f;
        for (int j = 0; j < I; ++j) {
          double g = c[j], u = c[I + j];
          hb[j] = oracle_bf16_round(g / (1.0 + exp(-g)) * u);
          float v = fabsf(bf16_to_f32(hb[j]));
          if (v > amax2) amax2 = v;
        }
        float sa2 = fmaxf(amax2, 1e-10f) / 448.0f;
        for (int j = 0; j < I; ++j)
          h2[j] = g_e4m3_lut[oracle_e4m3_encode(bf16_to_f32(hb[j]) / sa2)];
        const uint8_t* W2e = w2 + (int64_t)e * H * I;
        double wk = k < K ? (double)w[k] : 1.0;
        for (int cc = 0; cc < H; ++cc) {
          const uint8_t* b = W2e + (int64_t)cc * I;
          double acc = 0.0;
          for (int j = 0; j < I; ++j) acc += h2[j] * g_e4m3_lut[b[j]];
          o[cc] += wk * (acc * (double)sa2 * (double)s2[(int64_t)e * H + cc]);
        }
      }
    }
    free(kv);
    free(gkv);
    free(s);
    free(a);
    free(c);
    free(hb);
    free(h2);
  }
  return status;
}

/* ------------------------------------------------------------------------
 * Block-quantised FP8 (DeepSeek-V3's checkpoint format; the group_k/group_n
 * path that "Fix one bug in the grouped-gemm triton kernel", sglang #6772,
 * Highlights, contrasts with the per-token path). Activations carry one fp32
 * scale per token per 128 consecutive channels, weights one per 128 x 128
 * block (output-channel block x input-channel block). Each 128-channel
 * partial sum is dequantised by its own pair of scales:
 *   C[r,n] = sum_kb ( sum_{k in kb} q[r,k] W[n,k] ) * sa[r,kb] * sb[n/128,kb]
 * Block quantisation uses the per-token rule on each 128-block:
 *   s = max(amax_block, 1e-10) / 448, q = e4m3(x / s).
 * ---------------------------------------------------------------------- */
#define QB 128

void oracle_block_quant(const uint16_t* x, int64_t R, int C, uint8_t* q, float* scale) {
  const int nb = C / QB;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    for (int b = 0; b < nb; ++b) {
      const uint16_t* blk = x + r * C + (int64_t)b * QB;
      float amax = 0.0f;
      for (int c = 0; c < QB; ++c) {
        float v = fabsf(bf16_to_f32(blk[c]));
        if (v > amax) amax = v;
      }
      float sc = fmaxf(amax, 1e-10f) / 448.0f;
      scale[r * nb + b] = sc;
      for (int c = 0; c < QB; ++c)
        q[r * C + (int64_t)b * QB + c] = oracle_e4m3_encode(bf16_to_f32(blk[c]) / sc);
    }
  }
}

void oracle_permute_quant_block(const uint16_t* x, const int32_t* topk_ids, int T, int H,
                                int E, int K, uint8_t* a_q, float* scale_a, int32_t* src2dst,
                                int32_t* offsets) {
  const int nb = H / QB;
  oracle_route(topk_ids, T, E, K, offsets, src2dst);
  uint8_t* q = (uint8_t*)malloc((size_t)T * H + 1);
  float* sc = (float*)malloc(sizeof(float) * ((size_t)T * nb + 1));
  oracle_block_quant(x, T, H, q, sc);
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      int64_t d = src2dst[(int64_t)t * K + k];
      memcpy(a_q + d * H, q + (int64_t)t * H, (size_t)H);
      memcpy(scale_a + d * nb, sc + (int64_t)t * nb, sizeof(float) * (size_t)nb);
    }
  }
  free(q);
  free(sc);
}

void oracle_grouped_gemm_block(const uint8_t* A, const float* scale_a, const uint8_t* B,
                               const float* scale_b, const int32_t* offsets, int M, int N,
                               int Kd, int E, double* C) {
  init_lut();
  const int KB = Kd / QB, NBk = N / QB;
  int32_t* row_e = (int32_t*)malloc(sizeof(int32_t) * (size_t)(M > 0 ? M : 1));
  for (int r = 0; r < M; ++r) row_e[r] = -1;
  for (int e = 0; e < E; ++e)
    for (int r = offsets[e]; r < offsets[e + 1] && r < M; ++r) row_e[r] = e;
#pragma omp parallel
  {
    double* a = (double*)malloc(sizeof(double) * (size_t)Kd);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < M; ++r) {
      int e = row_e[r];
      double* c = C + (int64_t)r * N;
      if (e < 0) {
        for (int n = 0; n < N; ++n) c[n] = 0.0;
        continue;
      }
      for (int k = 0; k < Kd; ++k) a[k] = g_e4m3_lut[A[(int64_t)r * Kd + k]];
      const uint8_t* Be = B + (int64_t)e * N * Kd;
      const float* sbe = scale_b + (int64_t)e * NBk * KB;
      for (int n = 0; n < N; ++n) {
        const uint8_t* b = Be + (int64_t)n * Kd;
        double acc = 0.0;
        for (int kb = 0; kb < KB; ++kb) {
          double part = 0.0;
          for (int k = kb * QB; k < (kb + 1) * QB; ++k) part += a[k] * g_e4m3_lut[b[k]];
          acc += part * (double)scale_a[(int64_t)r * KB + kb] *
                 (double)sbe[(int64_t)(n / QB) * KB + kb];
        }
        c[n] = acc;
      }
    }
    free(a);
  }
  free(row_e);
}

/* Whole layer with block-quantised FP8 for the listed tokens, with n_shared
 * shared experts as in oracle_forward_tokens_shared. s13 [E+S, 2I/128, H/128],
 * s2 [E+S, H/128, I/128]. */
int oracle_forward_tokens_block(const uint16_t* x, const float* logits, const float* bias,
                                const uint8_t* w13, const float* s13, const uint8_t* w2,
                                const float* s2, int T, int H, int I, int E, int n_shared,
                                int num_groups, int topk_group, int top_k, int scoring,
                                int renormalize, float routed_scaling_factor,
                                const int64_t* tokens, int n_tok, double* out,
                                int32_t* ids_out, float* w_out) {
  int rc = gate_check(T, E, num_groups, topk_group, top_k, scoring, bias);
  if (rc) return rc;
  if (n_shared < 0 || H % QB != 0 || I % QB != 0) return -1;
  for (int i = 0; i < n_tok; ++i)
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
  init_lut();
  const int K = top_k;
  const int N13 = 2 * I;
  const int KBH = H / QB, KBI = I / QB;
  int status = 0;
#pragma omp parallel
  {
    kv_t* kv = (kv_t*)malloc(sizeof(kv_t) * (size_t)E);
    kv_t* gkv = (kv_t*)malloc(sizeof(kv_t) * (size_t)(E + num_groups));
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    float* sa = (float*)malloc(sizeof(float) * (size_t)KBH);
    double* c = (double*)malloc(sizeof(double) * (size_t)N13);
    uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    double* h2 = (double*)malloc(sizeof(double) * (size_t)I);
    float* sa2 = (float*)malloc(sizeof(float) * (size_t)KBI);
    int32_t ids[64];
    float w[64];
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < n_tok; ++i) {
      int64_t t = tokens[i];
      double* o = out + (int64_t)i * H;
      if (K > 64) {
        status = -2;
        continue;
      }
      gate_token(logits + t * E, bias, E, num_groups, topk_group, K, scoring, renormalize,
                 routed_scaling_factor, ids, w, kv, gkv, s);
      if (ids_out)
        for (int k = 0; k < K; ++k) ids_out[(int64_t)i * K + k] = ids[k];
      if (w_out)
        for (int k = 0; k < K; ++k) w_out[(int64_t)i * K + k] = w[k];
      /* block quantisation of the hidden state: one scale per 128 channels */
      const uint16_t* xr = x + t * H;
      for (int b = 0; b < KBH; ++b) {
        float amax = 0.0f;
        for (int hh = b * QB; hh < (b + 1) * QB; ++hh) {
          float v = fabsf(bf16_to_f32(xr[hh]));
          if (v > amax) amax = v;
        }
        sa[b] = fmaxf(amax, 1e-10f) / 448.0f;
        for (int hh = b * QB; hh < (b + 1) * QB; ++hh)
          a[hh] = g_e4m3_lut[oracle_e4m3_encode(bf16_to_f32(xr[hh]) / sa[b])];
      }
      for (int cc = 0; cc < H; ++cc) o[cc] = 0.0;
      for (int k = 0; k < K + n_shared; ++k) {
        const int e = k < K ? ids[k] : E + (k - K);
        const uint8_t* We = w13 + (int64_t)e * N13 * H;
        const float* sbe = s13 + (int64_t)e * (N13 / QB) * KBH;
        for (int n = 0; n < N13; ++n) {
          const uint8_t* b = We + (int64_t)n * H;
          double acc = 0.0;
          for (int kb = 0; kb < KBH; ++kb) {
            double part = 0.0;
            for (int hh = kb * QB; hh < (kb + 1) * QB; ++hh) part += a[hh] * g_e4m3_lut[b[hh]];
            acc += part * (double)sa[kb] * (double)sbe[(int64_t)(n / QB) * KBH + kb];
          }
          c[n] = acc;
        }
        for (int j = 0; j < I; ++j) {
          double g = c[j], u = c[I + j];
          hb[j] = oracle_bf16_round(g / (1.0 + exp(-g)) * u);
        }
        /* block requantisation of h */
        for (int b = 0; b < KBI; ++b) {
          float amax2 = 0.0f;
          for (int j = b * QB; j < (b + 1) * QB; ++j) {
            float v = fabsf(bf16_to_f32(hb[j]));
            if (v > amax2) amax2 = v;
          }
          sa2[b] = fmaxf(amax2, 1e-10f) / 448.0f;
          for (int j = b * QB; j < (b + 1) * QB; ++j)
            h2[j] = g_e4m3_lut[oracle_e4m3_encode(bf16_to_f32(hb[j]) / sa2[b])];
        }
        const uint8_t* W2e = w2 + (int64_t)e * H * I;
        const float* sb2 = s2 + (int64_t)e * (H / QB) * KBI;
        double wk = k < K ? (double)w[k] : 1.0;
        for (int cc = 0; cc < H; ++cc) {
          const uint8_t* b = W2e + (int64_t)cc * I;
          double acc = 0.0;
          for (int kb = 0; kb < KBI; ++kb) {
            double part = 0.0;
            for (int j = kb * QB; j < (kb + 1) * QB; ++j) part += h2[j] * g_e4m3_lut[b[j]];
            acc += part * (double)sa2[kb] * (double)sb2[(int64_t)(cc / QB) * KBI + kb];
          }
          o[cc] += wk * acc;
        }
      }
    }
    free(kv);
    free(gkv);
    free(s);
    free(a);
    free(sa);
    free(c);
    free(hb);
    free(h2);
    free(sa2);
  }
  return status;
}

/* ------------------------------------------------------------------------
 * NVFP4: the FP4 format the pages deploy DeepSeek-R1 in (modelopt_fp4 and
 * ModelOptNvFp4FusedMoEMethod, "[1/2] sgl-kernel: Fuse routed scaling factor
 * into select_experts", sglang #8364, Motivation and Highlights). The pages
 * name the format without writing it out. Reading, from NVIDIA's published
 * NVFP4 description:
 *  - elements are E2M1 codes (sign bit, 2 exponent bits with bias 1, one
 *    mantissa bit): magnitudes 0, 0.5 (the one subnormal), 1, 1.5, 2, 3, 4,
 *    6; encoding rounds to nearest with ties to the even code and saturates
 *    to +-6;
 *  - every 16 consecutive elements along K share one E4M3 block scale;
 *  - the tensor has one fp32 global scale g (an input: for weights it ships
 *    with the checkpoint, for activations it is the calibrated input scale);
 *  - value = e2m1(q) * e4m3(sb) * g.
 * Quantising a block: sb = e4m3((amax / 6) / g) (fp32 operations), then
 * q = e2m1(x / (e4m3(sb) * g)); a block whose scale decodes to 0 gets zero
 * codes. Codes are kept one per byte here (values 0..15).
 * ---------------------------------------------------------------------- */
#define FB 16

double oracle_e2m1_decode(uint8_t q) {
  int s = (q >> 3) & 1;
  int e = (q >> 1) & 3;
  int m = q & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

uint8_t oracle_e2m1_encode(float x) {
  uint32_t bits;
  memcpy(&bits, &x, 4);
  uint8_t sign = (bits >> 31) ? 0x8 : 0x0;
  float a = fabsf(x);
  if (a >= 6.0f) return (uint8_t)(sign | 0x7); /* saturate (also +-inf) */
  if (a < 1.0f) {
    /* subnormal range: units of 0.5; m == 2 is the smallest normal, 1.0,
     * whose code is also 2 */
    int m = (int)rintf(a * 2.0f); /* exact scaling */
    return (uint8_t)(sign | m);
  }
  int ex;
  frexpf(a, &ex);
  int E = ex - 1;                 /* a in [2^E, 2^(E+1)), E in 0..2 */
  float u = ldexpf(a, 1 - E);     /* units of the ulp 2^(E-1): u in [2, 4) */
  int m = (int)rintf(u);
  if (m == 4) {
    m = 2;
    E += 1;
  }
  int code = ((E + 1) << 1) | (m - 2);
  if (code > 0x7) code = 0x7;
  return (uint8_t)(sign | code);
}

void oracle_e2m1_encode_n(const float* x, uint8_t* q, int64_t n) {
  for (int64_t i = 0; i < n; ++i) q[i] = oracle_e2m1_encode(x[i]);
}

/* one bf16 row of C values (C % 16 == 0) -> C E2M1 codes, C/16 E4M3 codes */
static void nvfp4_quant_row(const uint16_t* row, int C, float g, uint8_t* q, uint8_t* sb) {
  for (int b = 0; b < C / FB; ++b) {
    const uint16_t* blk = row + (int64_t)b * FB;
    float amax = 0.0f;
    for (int c = 0; c < FB; ++c) {
      float v = fabsf(bf16_to_f32(blk[c]));
      if (v > amax) amax = v;
    }
    uint8_t s = oracle_e4m3_encode((amax / 6.0f) / g);
    sb[b] = s;
    float step = (float)oracle_e4m3_decode(s) * g;
    for (int c = 0; c < FB; ++c)
      q[(int64_t)b * FB + c] = step > 0.0f ? oracle_e2m1_encode(bf16_to_f32(blk[c]) / step) : 0;
  }
}

void oracle_nvfp4_quant(const uint16_t* x, int64_t R, int C, float g, uint8_t* q,
                        uint8_t* sb) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) nvfp4_quant_row(x + r * C, C, g, q + r * C, sb + r * (C / FB));
}

void oracle_grouped_gemm_nvfp4(const uint8_t* A, const uint8_t* sa, float ga, const uint8_t* B,
                               const uint8_t* sb, const float* gb, const int32_t* offsets,
                               int M, int N, int Kd, int E, double* C) {
  init_lut();
  const int KB = Kd / FB;
  int32_t* row_e = (int32_t*)malloc(sizeof(int32_t) * (size_t)(M > 0 ? M : 1));
  for (int r = 0; r < M; ++r) row_e[r] = -1;
  for (int e = 0; e < E; ++e)
    for (int r = offsets[e]; r < offsets[e + 1] && r < M; ++r) row_e[r] = e;
#pragma omp parallel
  {
    double* a = (double*)malloc(sizeof(double) * (size_t)Kd);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < M; ++r) {
      int e = row_e[r];
      double* c = C + (int64_t)r * N;
      if (e < 0) {
        for (int n = 0; n < N; ++n) c[n] = 0.0;
        continue;
      }
      for (int k = 0; k < Kd; ++k) a[k] = oracle_e2m1_decode(A[(int64_t)r * Kd + k]);
      const uint8_t* Be = B + (int64_t)e * N * Kd;
      const uint8_t* sbe = sb + (int64_t)e * N * KB;
      for (int n = 0; n < N; ++n) {
        const uint8_t* b = Be + (int64_t)n * Kd;
        double acc = 0.0;
        for (int kb = 0; kb < KB; ++kb) {
          double part = 0.0; /* exact: products are multiples of 1/4 below 37 */
          for (int k = kb * FB; k < (kb + 1) * FB; ++k) part += a[k] * oracle_e2m1_decode(b[k]);
          acc += part * g_e4m3_lut[sa[(int64_t)r * KB + kb]] *
                 g_e4m3_lut[sbe[(int64_t)n * KB + kb]];
        }
        c[n] = acc * (double)ga * (double)gb[e];
      }
    }
    free(a);
  }
  free(row_e);
}

/* The whole layer in NVFP4 for the listed tokens, with n_shared shared
 * experts as in oracle_forward_tokens_shared: the hidden state is quantised
 * with the input global scale ga1, h (rounded to bf16) with ga2, and each
 * expert's weights carry their own global scales g13[e], g2[e]. Weight
 * codes w13 [E+S,2I,H], w2 [E+S,H,I]; block scales s13 [E+S,2I,H/16],
 * s2 [E+S,H,I/16] (E4M3 codes). */
int oracle_forward_tokens_nvfp4(const uint16_t* x, const float* logits, const float* bias,
                                const uint8_t* w13, const uint8_t* s13, const float* g13,
                                const uint8_t* w2, const uint8_t* s2, const float* g2,
                                float ga1, float ga2, int T, int H, int I, int E,
                                int n_shared, int num_groups, int topk_group, int top_k,
                                int scoring, int renormalize, float routed_scaling_factor,
                                const int64_t* tokens, int n_tok, double* out,
                                int32_t* ids_out, float* w_out) {
  int rc = gate_check(T, E, num_groups, topk_group, top_k, scoring, bias);
  if (rc) return rc;
  if (n_shared < 0 || H % FB != 0 || I % FB != 0 || !(ga1 > 0.0f) || !(ga2 > 0.0f)) return -1;
  for (int i = 0; i < n_tok; ++i)
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
  init_lut();
  const int K = top_k;
  const int N13 = 2 * I;
  const int KBH = H / FB, KBI = I / FB;
  int status = 0;
#pragma omp parallel
  {
    kv_t* kv = (kv_t*)malloc(sizeof(kv_t) * (size_t)E);
    kv_t* gkv = (kv_t*)malloc(sizeof(kv_t) * (size_t)(E + num_groups));
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    uint8_t* qa = (uint8_t*)malloc((size_t)H);
    uint8_t* sa = (uint8_t*)malloc((size_t)KBH);
    double* c = (double*)malloc(sizeof(double) * (size_t)N13);
    uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    uint8_t* q2 = (uint8_t*)malloc((size_t)I);
    uint8_t* sa2 = (uint8_t*)malloc((size_t)KBI);
    int32_t ids[64];
    float w[64];
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < n_tok; ++i) {
      int64_t t = tokens[i];
      double* o = out + (int64_t)i * H;
      if (K > 64) {
        status = -2;
        continue;
      }
      gate_token(logits + t * E, bias, E, num_groups, topk_group, K, scoring, renormalize,
                 routed_scaling_factor, ids, w, kv, gkv, s);
      if (ids_out)
        for (int k = 0; k < K; ++k) ids_out[(int64_t)i * K + k] = ids[k];
      if (w_out)
        for (int k = 0; k < K; ++k) w_out[(int64_t)i * K + k] = w[k];
      nvfp4_quant_row(x + t * H, H, ga1, qa, sa);
      for (int cc = 0; cc < H; ++cc) o[cc] = 0.0;
      for (int k = 0; k < K + n_shared; ++k) {
        const int e = k < K ? ids[k] : E + (k - K);
        const uint8_t* We = w13 + (int64_t)e * N13 * H;
        const uint8_t* sbe = s13 + (int64_t)e * N13 * KBH;
        for (int n = 0; n < N13; ++n) {
          const uint8_t* b = We + (int64_t)n * H;
          double acc = 0.0;
          for (int kb = 0; kb < KBH; ++kb) {
            double part = 0.0;
            for (int hh = kb * FB; hh < (kb + 1) * FB; ++hh)
              part += oracle_e2m1_decode(qa[hh]) * oracle_e2m1_decode(b[hh]);
            acc += part * g_e4m3_lut[sa[kb]] * g_e4m3_lut[sbe[(int64_t)n * KBH + kb]];
          }
          c[n] = acc * (double)ga1 * (double)g13[e];
        }
        for (int j = 0; j < I; ++j) {
          double g = c[j], u = c[I + j];
          hb[j] = oracle_bf16_round(g / (1.0 + exp(-g)) * u);
        }
        nvfp4_quant_row(hb, I, ga2, q2, sa2);
        const uint8_t* W2e = w2 + (int64_t)e * H * I;
        const uint8_t* sb2 = s2 + (int64_t)e * H * KBI;
        double wk = k < K ? (double)w[k] : 1.0;
        for (int cc = 0; cc < H; ++cc) {
          const uint8_t* b = W2e + (int64_t)cc * I;
          double acc = 0.0;
          for (int kb = 0; kb < KBI; ++kb) {
            double part = 0.0;
            for (int j = kb * FB; j < (kb + 1) * FB; ++j)
              part += oracle_e2m1_decode(q2[j]) * oracle_e2m1_decode(b[j]);
            acc += part * g_e4m3_lut[sa2[kb]] * g_e4m3_lut[sb2[(int64_t)cc * KBI + kb]];
          }
          o[cc] += wk * (acc * (double)ga2 * (double)g2[e]);
        }
      }
    }
    free(kv);
    free(gkv);
    free(s);
    free(qa);
    free(sa);
    free(c);
    free(hb);
    free(q2);
    free(sa2);
  }
  return status;
}
