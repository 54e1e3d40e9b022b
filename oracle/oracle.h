/*
 * Oracle for the grouped-expert MoE layer forward: plain, slow, CPU-only C.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library. The product path (the
 * CUDA library) never links, loads or calls it, and shares no code with it.
 *
 * What it computes follows three sglang pull-request pages:
 *   - "Fix one bug in the grouped-gemm triton kernel" (sglang #6772),
 *     Highlights: scale_a is indexed by row (m_range_start + offs_am), not by
 *     the expert id, when block quantisation is off.
 *   - "Support token-level quantization for EP MoE" (sglang #6782), Summary of
 *     Changes / Changelog: per-token dynamic FP8 activation scales, loaded per
 *     token in the pre-reorder kernel and in the grouped GEMM, reordered via
 *     src2dst, and the activation output requantised per token.
 *   - "[1/2] sgl-kernel: Fuse routed scaling factor into select_experts"
 *     (sglang #8364), Motivation / Highlights: routed_scaling_factor is
 *     multiplied into the renormalised top-k weights inside the gate.
 * Steps the pages leave open are fixed by the readings listed in each
 * function's comment.
 *
 * Precision: fp64 everywhere the method does not fix a precision, except
 * where floating point decides an integer (top-k ids, FP8 codes): those
 * decisions are taken in fp32, the precision of the kernel, with IEEE
 * single-precision operations written out one by one (this file must be
 * compiled with -ffp-contract=off).
 *
 * Layouts (all row-major, element sizes in brackets):
 *   logits [T,E] f32, bias [E] f32 (may be NULL), topk_ids [T,K] i32,
 *   topk_w [T,K] f32, x [T,H] bf16 bits (u16), a_q [M,H] e4m3 (u8),
 *   scale_a [M] f32, src2dst [T*K] i32, offsets [E+1] i32,
 *   w13 [E,2I,H] e4m3 with rows 0..I-1 the gate projection and I..2I-1 the
 *   up projection, s13 [E,2I] f32, w2 [E,H,I] e4m3, s2 [E,H] f32.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Scoring functions of the gate. */
enum { ORACLE_SIGMOID = 0, ORACLE_SOFTMAX = 1 };

void oracle_set_threads(int n);
int oracle_get_threads(void);

/* fp32 exponential: Cody-Waite reduction + degree-7 Taylor polynomial. */
float oracle_exp32(float x);
void oracle_exp32_n(const float* x, float* y, int64_t n);
/* fp32 logistic function 1 / (1 + exp(-x)). */
float oracle_sigmoid32(float x);
void oracle_sigmoid32_n(const float* x, float* y, int64_t n);

/* OCP FP8 e4m3 (fn): round to nearest even, saturate to +-448. */
uint8_t oracle_e4m3_encode(float x);
void oracle_e4m3_encode_n(const float* x, uint8_t* q, int64_t n);
double oracle_e4m3_decode(uint8_t q);

/* fp64 -> bf16 bits, round to nearest even (single rounding). */
uint16_t oracle_bf16_round(double v);
void oracle_bf16_round_n(const double* v, uint16_t* out, int64_t n);

/* Gate. Returns 0, or -1 for invalid arguments, -2 for unsupported ones. */
int oracle_gate(const float* logits, const float* bias, int T, int E,
                int num_groups, int topk_group, int top_k, int scoring,
                int renormalize, float routed_scaling_factor,
                int32_t* topk_ids, float* topk_w);

/* Stable counting sort of the flattened (token, slot) pairs by expert. */
void oracle_route(const int32_t* topk_ids, int T, int E, int K,
                  int32_t* offsets, int32_t* src2dst);

/* Per-row dynamic FP8 quantisation of a bf16 matrix [R,C]. */
void oracle_row_quant(const uint16_t* x, int64_t R, int C, uint8_t* q,
                      float* scale);

/* Route + quantise each token once + scatter its codes and scale to the K
 * destinations (pre-reorder). */
void oracle_permute_quant(const uint16_t* x, const int32_t* topk_ids, int T,
                          int H, int E, int K, uint8_t* a_q, float* scale_a,
                          int32_t* src2dst, int32_t* offsets);

/* Grouped GEMM: C[r,n] = (sum_k A[r,k] B[e,n,k]) * scale_a[r] * scale_b[e,n]
 * for r in expert e's segment, in fp64. */
void oracle_grouped_gemm(const uint8_t* A, const float* scale_a,
                         const uint8_t* B, const float* scale_b,
                         const int32_t* offsets, int M, int N, int Kd, int E,
                         double* C);

/* h[r,j] = silu(C[r,j]) * C[r,I+j] in fp64. */
void oracle_silu_mul(const double* C, int64_t M, int I, double* h);

/* out[t,:] = sum_k w[t,k] * down[src2dst[t*K+k], :] in fp64. */
void oracle_unpermute_sum(const double* down, const int32_t* src2dst,
                          const float* topk_w, int T, int K, int H,
                          double* out);

/* Whole layer for the tokens listed in `tokens` (n_tok of them; each token's
 * output depends on that token alone). out [n_tok,H] fp64. Also returns the
 * gate result of those tokens when ids_out / w_out are non-NULL. */
int oracle_forward_tokens(const uint16_t* x, const float* logits,
                          const float* bias, const uint8_t* w13,
                          const float* s13, const uint8_t* w2, const float* s2,
                          int T, int H, int I, int E, int num_groups,
                          int topk_group, int top_k, int scoring,
                          int renormalize, float routed_scaling_factor,
                          const int64_t* tokens, int n_tok, double* out,
                          int32_t* ids_out, float* w_out);

/* The same with n_shared shared experts stored as experts E .. E+n_shared-1
 * of w13 [E+n_shared,2I,H] / w2 [E+n_shared,H,I] (scales likewise): each
 * token adds every shared expert's output with weight 1 after its K routed
 * experts. The gate sees only the E routed experts. */
int oracle_forward_tokens_shared(const uint16_t* x, const float* logits,
                                 const float* bias, const uint8_t* w13,
                                 const float* s13, const uint8_t* w2, const float* s2,
                                 int T, int H, int I, int E, int n_shared,
                                 int num_groups, int topk_group, int top_k, int scoring,
                                 int renormalize, float routed_scaling_factor,
                                 const int64_t* tokens, int n_tok, double* out,
                                 int32_t* ids_out, float* w_out);

/* ---- block-quantised FP8 (128-channel activation blocks, 128 x 128 weight
 * blocks; every dimension that is blocked must be a multiple of 128) ---- */

/* x bf16 [R,C] -> q e4m3 [R,C], scale f32 [R, C/128]: per 128-block of a row,
 * scale = max(amax, 1e-10)/448, q = e4m3(x / scale). */
void oracle_block_quant(const uint16_t* x, int64_t R, int C, uint8_t* q, float* scale);

/* oracle_permute_quant with block scales: scale_a [T*K, H/128]. */
void oracle_permute_quant_block(const uint16_t* x, const int32_t* topk_ids, int T, int H,
                                int E, int K, uint8_t* a_q, float* scale_a, int32_t* src2dst,
                                int32_t* offsets);

/* C[r,n] = sum_kb (sum_{k in kb} A[r,k] B[e,n,k]) * scale_a[r,kb] *
 * scale_b[e, n/128, kb] in fp64. scale_a [M, Kd/128]; scale_b [E, N/128, Kd/128]. */
void oracle_grouped_gemm_block(const uint8_t* A, const float* scale_a, const uint8_t* B,
                               const float* scale_b, const int32_t* offsets, int M, int N,
                               int Kd, int E, double* C);

/* The whole layer in block FP8 (with n_shared shared experts as in
 * oracle_forward_tokens_shared). s13 [E+S, 2I/128, H/128]; s2 [E+S, H/128, I/128]. */
int oracle_forward_tokens_block(const uint16_t* x, const float* logits, const float* bias,
                                const uint8_t* w13, const float* s13, const uint8_t* w2,
                                const float* s2, int T, int H, int I, int E, int n_shared,
                                int num_groups, int topk_group, int top_k, int scoring,
                                int renormalize, float routed_scaling_factor,
                                const int64_t* tokens, int n_tok, double* out,
                                int32_t* ids_out, float* w_out);

/* NVFP4 (E2M1 elements, one E4M3 scale per 16 elements along K, one fp32
 * global scale per tensor). Codes one per byte (0..15). */
double oracle_e2m1_decode(uint8_t q);
/* nearest E2M1 code, ties to the even code, saturating to +-6 */
uint8_t oracle_e2m1_encode(float x);
void oracle_e2m1_encode_n(const float* x, uint8_t* q, int64_t n);

/* x bf16 [R,C] (C % 16 == 0), global scale g > 0 -> q [R,C] E2M1 codes,
 * sb [R, C/16] E4M3 block-scale codes: sb = e4m3((amax/6)/g),
 * q = e2m1(x / (e4m3(sb) * g)), zero codes where the scale decodes to 0. */
void oracle_nvfp4_quant(const uint16_t* x, int64_t R, int C, float g, uint8_t* q,
                        uint8_t* sb);

/* C[r,n] = ga * gb[e] * sum_kb (sum_{k in kb} e2m1(A[r,k]) e2m1(B[e,n,k])) *
 * e4m3(sa[r,kb]) * e4m3(sb[e,n,kb]) in fp64, kb the 16-element blocks of K.
 * A [M,Kd], sa [M,Kd/16], B [E,N,Kd], sb [E,N,Kd/16], gb [E]. */
void oracle_grouped_gemm_nvfp4(const uint8_t* A, const uint8_t* sa, float ga, const uint8_t* B,
                               const uint8_t* sb, const float* gb, const int32_t* offsets,
                               int M, int N, int Kd, int E, double* C);

/* The whole layer in NVFP4 (with n_shared shared experts as in
 * oracle_forward_tokens_shared): x quantised with the global scale ga1, the
 * bf16-rounded h with ga2; w13 [E+S,2I,H] and w2 [E+S,H,I] E2M1 codes,
 * s13 [E+S,2I,H/16] and s2 [E+S,H,I/16] E4M3 block-scale codes, g13 and g2
 * [E+S] the weights' global scales. H % 16 == 0, I % 16 == 0. */
int oracle_forward_tokens_nvfp4(const uint16_t* x, const float* logits, const float* bias,
                                const uint8_t* w13, const uint8_t* s13, const float* g13,
                                const uint8_t* w2, const uint8_t* s2, const float* g2,
                                float ga1, float ga2, int T, int H, int I, int E,
                                int n_shared, int num_groups, int topk_group, int top_k,
                                int scoring, int renormalize, float routed_scaling_factor,
                                const int64_t* tokens, int n_tok, double* out,
                                int32_t* ids_out, float* w_out);

#ifdef __cplusplus
}
#endif
#endif
