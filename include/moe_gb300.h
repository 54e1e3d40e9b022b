/*
 * moe_gb300: forward pass of a grouped-expert Mixture-of-Experts layer with
 * all experts on one GB300 (sm_103a), as a C ABI.
 *
 * The layer follows three sglang pull-request pages:
 *   [P1] "Fix one bug in the grouped-gemm triton kernel" (sglang #6772)
 *   [P2] "Support token-level quantization for EP MoE" (sglang #6782)
 *   [P3] "[1/2] sgl-kernel: Fuse routed scaling factor into select_experts"
 *        (sglang #8364)
 * Steps, in order: grouped top-k gate with routed_scaling_factor fused in
 * (moe_gate), pre-reorder with per-token FP8 quantisation
 * (moe_permute_quant), w13 grouped GEMM with per-row scale_a and
 * per-channel scale_b plus SiLU*mul (moe_grouped_gemm), per-token
 * requantisation (moe_act_quant), w2 grouped GEMM (moe_grouped_gemm) and
 * the weighted post-reorder (moe_unpermute_sum); moe_forward runs them all.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless the name ends in _host. The caller
 *    owns every buffer; no entry point allocates device memory per call.
 *    (The library keeps, per device, a 4-byte error word it allocates at
 *    load time as a static device variable.)
 *  - bf16 tensors are passed as void* to 16-bit bfloat16 values, FP8 tensors
 *    as void* to 8-bit OCP e4m3 ("e4m3fn": bias 7, max 448, no inf) codes.
 *  - All tensors are dense, row-major, with the last dimension contiguous.
 *    Every tensor pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL: the legacy default stream). Every call
 *    is asynchronous on that stream and never synchronises the host.
 *  - Errors are returned as moe_status codes and never thrown. Arguments are
 *    validated on the host before anything is launched; an invalid call
 *    launches nothing. MOE_ERR_CUDA means a launch failed (the CUDA error is
 *    left for cudaGetLastError). Faults detected inside a kernel (an expert
 *    id out of range, a pipeline wait that timed out) set the device error
 *    word; read and clear it with moe_device_status().
 *  - Inputs containing NaN or Inf are outside the contract.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* a size, pointer or alignment is invalid */
  MOE_ERR_UNSUPPORTED = -2, /* valid but outside what the kernels handle */
  MOE_ERR_WORKSPACE = -3,   /* workspace missing or too small */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE = -5       /* moe_device_status: a kernel flagged a fault */
} moe_status;

typedef enum { MOE_SCORE_SIGMOID = 0, MOE_SCORE_SOFTMAX = 1 } moe_scoring;

typedef enum {
  MOE_EPI_BF16 = 0,    /* C[r,n] = bf16(acc * scale_a[r] * scale_b[e,n]) */
  MOE_EPI_SILU_MUL = 1 /* h[r,j] = bf16(silu(C[r,j]) * C[r,I+j]), I = N/2 */
} moe_epilogue;

/* Device-side fault codes reported by moe_device_status(). */
enum {
  MOE_DEV_OK = 0,
  MOE_DEV_BAD_EXPERT_ID = 1,  /* moe_permute_quant: topk_ids out of [0,E) */
  MOE_DEV_PIPE_TIMEOUT = 2,   /* moe_grouped_gemm: a pipeline wait gave up */
  MOE_DEV_BAD_OFFSETS = 3     /* moe_grouped_gemm: offsets not monotone or > M */
};

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(moe_status s);

/* Version of this ABI: (major << 16) | minor. */
MOE_API int moe_abi_version(void);

/*
 * moe_gate — grouped, bias-corrected top-k expert selection.
 * [P3] Motivation/Highlights: the selected experts' weights are normalised
 * and multiplied by routed_scaling_factor inside the gate; [P3] names the
 * biased grouped top-k op. Semantics (readings where the pages are silent):
 *   scoring SIGMOID: s = 1/(1+exp(-l)) (fp32, exp by Cody-Waite reduction and
 *     a degree-7 Taylor polynomial); key b = s + bias[e] (bias NULL: 0).
 *     Group g (experts [g*E/G, (g+1)*E/G)) scores the sum of its two largest
 *     keys (its only key for one-expert groups); the topk_group best groups
 *     are kept; the top_k largest keys among the kept groups are selected.
 *     Ties go to the lower index. Slot k holds the k-th selection.
 *     Weights: w_k = s_k / S * rsf with S the fp32 slot-order sum of the
 *     selected s (renormalize != 0), or w_k = s_k * rsf.
 *   scoring SOFTMAX (requires bias == NULL and num_groups == 1): experts are
 *     selected by logit; w_k = exp(l_k - l_slot0) / S * rsf (renormalize), or
 *     exp(l_k - l_max) / Z * rsf with Z summed over all experts in order.
 * logits [T,E] f32; bias [E] f32 or NULL; topk_ids [T,top_k] i32 (out);
 * topk_w [T,top_k] f32 (out). Bit-exact across runs.
 * Limits: 1 <= E <= 1024, E % num_groups == 0, num_groups <= 64,
 * 1 <= topk_group <= num_groups, 1 <= top_k <= min(32, topk_group*E/G).
 */
MOE_API moe_status moe_gate(const float* logits, const float* bias, int T, int E,
                    int num_groups, int topk_group, int top_k, int scoring,
                    int renormalize, float routed_scaling_factor,
                    int32_t* topk_ids, float* topk_w, void* stream);

/* Workspace bytes moe_permute_quant needs for T tokens, E experts. */
MOE_API size_t moe_permute_workspace_size(int T, int E, int K);

/*
 * moe_permute_quant — pre-reorder with dynamic per-token FP8 quantisation.
 * [P2] Summary/Changelog: per-token activation scales from per-token maxima,
 * loaded per token in the pre-reorder; the scales are written in permuted
 * order through src2dst ([P2] Code Review). [P1] Highlights: each expert
 * owns a contiguous row range starting at m_range_start.
 *   Routing: the flattened pairs i = t*K + k are counting-sorted by expert,
 *   stable in i (so ascending t within an expert): offsets[0] = 0,
 *   offsets[e+1] = offsets[e] + count[e]; src2dst[i] = destination row.
 *   Quantisation of token t: amax = max|x[t,:]|, scale = max(amax,1e-10)/448
 *   (fp32), code = e4m3_rne_satfinite(x / scale) (IEEE division);
 *   a_q[src2dst[t*K+k], :] = codes and scale_a[src2dst[t*K+k]] = scale for
 *   every slot k.
 * x [T,H] bf16; topk_ids [T,K] i32 (values in [0,E), distinct per token);
 * a_q [T*K,H] e4m3 (out); scale_a [T*K] f32 (out); src2dst [T*K] i32 (out);
 * offsets [E+1] i32 (out); ws: moe_permute_workspace_size(T,E,K) bytes,
 * 256-byte aligned (contents on entry ignored). Bit-exact.
 * Limits: H % 32 == 0, 1 <= E <= 1024, 1 <= K <= 32, T*K < 2^31.
 */
MOE_API moe_status moe_permute_quant(const void* x, const int32_t* topk_ids, int T,
                             int H, int E, int K, void* a_q, float* scale_a,
                             int32_t* src2dst, int32_t* offsets, void* ws,
                             size_t ws_bytes, void* stream);

/* Size of the fixed device scratch behind moe_permute_quant_noalloc. */
#define MOE_PERMUTE_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/*
 * moe_permute_quant_noalloc — moe_permute_quant without a workspace argument.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory and have no workspace to hand over, such as
 * code running as a plug-in inside another runtime that owns all device
 * memory and passes it only its input and output buffers, or code on a
 * latency-critical path where an allocation (which can synchronise the
 * device) is not acceptable. It computes exactly what moe_permute_quant
 * computes, with the same arguments minus ws / ws_bytes.
 *   Scratch: a fixed array of MOE_PERMUTE_NOALLOC_SCRATCH_BYTES (4 MiB) in
 *   the library's device memory, reserved on every GPU that loads the
 *   library until the process exits. The call needs
 *   moe_permute_workspace_size(T,E,K) <= MOE_PERMUTE_NOALLOC_SCRATCH_BYTES
 *   (e.g. T <= 65536 tokens at E = 256); larger sizes return
 *   MOE_ERR_WORKSPACE and launch nothing.
 *   Set-up: the first call on each device looks up the array's device
 *   address with that device current; make that first call before any
 *   stream capture.
 *   Sharing: every call uses the same array and leaves its contents behind.
 *   Nothing in it has to start at zero (a call writes every scratch entry it
 *   later reads). Calls that overlap on the GPU (different streams, or
 *   unordered calls from several threads) race on the array and produce
 *   wrong results: order them.
 *   It calls no cudaMalloc, cudaFree or other allocating routine.
 */
MOE_API moe_status moe_permute_quant_noalloc(const void* x, const int32_t* topk_ids, int T,
                                             int H, int E, int K, void* a_q, float* scale_a,
                                             int32_t* src2dst, int32_t* offsets,
                                             void* stream);

/*
 * moe_grouped_gemm — FP8 grouped GEMM over expert row segments, tcgen05.
 * [P1] Highlights and [P2] Changelog: within expert e's rows
 * [offsets[e], offsets[e+1]) the fp32 accumulator is dequantised by the
 * ROW's per-token scale_a times the weight scale; no block quantisation.
 *   acc[r,n] = sum_k A[r,k] * B[e,n,k]   (fp32 accumulate on tensor cores)
 *   epilogue MOE_EPI_BF16:     C [M,N] bf16 = acc * scale_a[r] * scale_b[e,n]
 *   epilogue MOE_EPI_SILU_MUL: with I = N/2, g = that value for n = j and
 *     u for n = I + j: C [M,I] bf16 = silu(g) * u; if row_amax != NULL it
 *     must hold zeros on entry and receives max_j |C[r,j]| (after bf16
 *     rounding) for every row.
 * A [M,Kd] e4m3 (rows grouped by expert); scale_a [M] f32;
 * B [E,N,Kd] e4m3 (K-major weights; for SILU_MUL rows 0..I-1 are the gate
 * projection and I..2I-1 the up projection); scale_b [E,N] f32;
 * offsets [E+1] i32 on the device (monotone, offsets[E] <= M). Rows beyond
 * offsets[E] are not written. No workspace.
 * Limits: Kd % 32 == 0, N % 32 == 0 (SILU_MUL: N % 64 == 0), E <= 1024.
 */
MOE_API moe_status moe_grouped_gemm(const void* A, const float* scale_a,
                            const void* B, const float* scale_b,
                            const int32_t* offsets, int M, int N, int Kd,
                            int E, int epilogue, void* C, float* row_amax,
                            void* stream);

/*
 * moe_permute_quant_rows — moe_permute_quant with each token's codes stored
 * ONCE, in token order: a_tok [T,H] e4m3 (row t = token t's codes), and
 * row_token [T*K] i32 (out) = the token of each permuted row
 * (row_token[src2dst[t*K+k]] = t). scale_a [T*K] (permuted order), src2dst
 * and offsets as moe_permute_quant; same workspace and limits. A token's
 * K copies are not written (the K-fold row write of the pre-reorder becomes
 * one), and moe_grouped_gemm_rows reads the rows through row_token.
 * Bit-exact.
 */
MOE_API moe_status moe_permute_quant_rows(const void* x, const int32_t* topk_ids, int T,
                                          int H, int E, int K, void* a_tok, float* scale_a,
                                          int32_t* src2dst, int32_t* row_token,
                                          int32_t* offsets, void* ws, size_t ws_bytes,
                                          void* stream);

/*
 * moe_grouped_gemm_rows — moe_grouped_gemm whose permuted row r of A is row
 * row_token[r] of the token-order A_tok [T,Kd] e4m3 (each tile's token rows
 * are gathered four at a time by TMA). Everything else, results included,
 * as moe_grouped_gemm on A[r] = A_tok[row_token[r]]: scale_a [M] stays in
 * permuted order. row_token values outside [0,T) read as zero rows.
 * Speed: on the DeepSeek-V3 prefill w13 shape (M = 65536 rows, 256 experts)
 * this measured 4.31 ms against 1.72 ms for moe_grouped_gemm on the K-fold
 * copies (the four-row gathers bound it), so moe_forward does not use it;
 * it serves callers short of memory for the K copies.
 */
MOE_API moe_status moe_grouped_gemm_rows(const void* A_tok, int T, const int32_t* row_token,
                                         const float* scale_a, const void* B,
                                         const float* scale_b, const int32_t* offsets, int M,
                                         int N, int Kd, int E, int epilogue, void* C,
                                         float* row_amax, void* stream);

/*
 * moe_act_quant — per-token requantisation of the activation output.
 * [P2] Changelog/Code Review: down_input is quantised per token to FP8 with
 * the per-token quantiser, giving w2_input_scale.
 *   amax = row_amax[r] if row_amax != NULL, else max_j |h[r,j]|;
 *   scale[r] = max(amax,1e-10)/448 (fp32); q[r,j] = e4m3_rne_satfinite(
 *   h[r,j] / scale[r]).
 * h [M,I] bf16; row_amax [M] f32 or NULL; q [M,I] e4m3 (out);
 * scale [M] f32 (out). Bit-exact. Limits: I % 32 == 0.
 */
MOE_API moe_status moe_act_quant(const void* h, const float* row_amax, int M, int I,
                         void* q, float* scale, void* stream);

/*
 * moe_unpermute_sum — weighted post-reorder back to token order.
 * [P3] Motivation names moe_sum_reduce, the weighted top-k sum.
 *   out[t,:] = bf16( sum_{k=0..K-1} topk_w[t,k] * down[src2dst[t*K+k], :] )
 * accumulated in fp32 in slot order.
 * down [M,H] bf16; src2dst [T*K] i32; topk_w [T,K] f32; out [T,H] bf16.
 * Limits: H % 8 == 0, 1 <= K <= 32.
 */
MOE_API moe_status moe_unpermute_sum(const void* down, const int32_t* src2dst,
                             const float* topk_w, int T, int K, int H,
                             void* out, void* stream);

/* Workspace bytes moe_forward / moe_forward_host need. */
MOE_API size_t moe_workspace_size(int T, int H, int I, int E, int K);

/*
 * moe_forward — the whole layer: gate, pre-reorder + quant, w13 GEMM with
 * SiLU*mul, requant, w2 GEMM, weighted post-reorder, on one stream.
 * x [T,H] bf16; logits [T,E] f32; bias [E] f32 or NULL;
 * w13 [E,2I,H] e4m3 (rows: gate then up); s13 [E,2I] f32;
 * w2 [E,H,I] e4m3; s2 [E,H] f32; out [T,H] bf16.
 * ws: moe_workspace_size(T,H,I,E,top_k) bytes, 256-byte aligned; it holds
 * every intermediate (ids, weights, permuted codes, h, ...).
 * Limits: those of the steps; H % 32 == 0 and I % 32 == 0.
 */
MOE_API moe_status moe_forward(const void* x, const float* logits, const float* bias,
                       const void* w13, const float* s13, const void* w2,
                       const float* s2, int T, int H, int I, int E,
                       int num_groups, int topk_group, int top_k, int scoring,
                       int renormalize, float routed_scaling_factor, void* out,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward_host — moe_forward with the per-step tensors in HOST memory:
 * x_host [T,H] bf16 and logits_host [T,E] f32 in, out_host [T,H] bf16 out,
 * all asynchronously on `stream` (the host buffers must stay valid until the
 * stream reaches the end of this call). When all three buffers are pinned
 * and mapped into the device's address space (cudaHostAlloc, or torch's
 * pin_memory, with unified addressing), the kernels read x and logits and
 * write out in host memory directly over the host link; otherwise x and
 * logits are copied into the workspace first and out is copied back (use
 * pinned memory for asynchrony). Same results either way. Weights, scales
 * and bias stay device pointers.
 */
MOE_API moe_status moe_forward_host(const void* x_host, const float* logits_host,
                            const float* bias, const void* w13,
                            const float* s13, const void* w2, const float* s2,
                            int T, int H, int I, int E, int num_groups,
                            int topk_group, int top_k, int scoring,
                            int renormalize, float routed_scaling_factor,
                            void* out_host, void* ws, size_t ws_bytes,
                            void* stream);

/*
 * moe_forward_shared — moe_forward plus n_shared shared experts, which every
 * token runs besides its top_k routed experts. [P3] Highlights (sglang
 * #8364) notes that shared-expert fusion works together with the scaling
 * factor fused into the gate; the pages give no formula, so this takes the
 * DeepSeek-V3 layer: out = sum_k w_k expert_k(x) + sum_j shared_j(x), the
 * shared experts with weight 1 (routed_scaling_factor is already in w_k).
 * Layout: the shared experts are experts E .. E+n_shared-1 of the weight
 * tensors, of the routed experts' size: w13 [E+n_shared,2I,H],
 * s13 [E+n_shared,2I], w2 [E+n_shared,H,I], s2 [E+n_shared,H]. logits and
 * bias cover the E routed experts only. The gate appends the shared slots
 * to each token's row and the rest of the layer runs as a routed layer of
 * E+n_shared experts and top_k+n_shared slots, summed in slot order.
 * ws: moe_workspace_size(T,H,I,E+n_shared,top_k+n_shared) bytes.
 * n_shared == 0 is moe_forward. Limits: E+n_shared <= 1024,
 * top_k+n_shared <= 32; otherwise those of moe_forward.
 */
MOE_API moe_status moe_forward_shared(const void* x, const float* logits,
                              const float* bias, const void* w13,
                              const float* s13, const void* w2, const float* s2,
                              int T, int H, int I, int E, int n_shared,
                              int num_groups, int topk_group, int top_k,
                              int scoring, int renormalize,
                              float routed_scaling_factor, void* out, void* ws,
                              size_t ws_bytes, void* stream);

/* moe_forward_shared with the per-step tensors in host memory, as
 * moe_forward_host. */
MOE_API moe_status moe_forward_shared_host(const void* x_host,
                              const float* logits_host, const float* bias,
                              const void* w13, const float* s13, const void* w2,
                              const float* s2, int T, int H, int I, int E,
                              int n_shared, int num_groups, int topk_group,
                              int top_k, int scoring, int renormalize,
                              float routed_scaling_factor, void* out_host,
                              void* ws, size_t ws_bytes, void* stream);

/* ==========================================================================
 * Block-quantised FP8: one fp32 scale per 128 x 128 weight block (output
 * block x input block) and one per token per 128 input channels, the format
 * DeepSeek-V3 checkpoints ship in. [P1] Highlights contrasts the per-token
 * path with this block (group_k / group_n) path; it does not write the
 * formula, taken here as: every 128-channel partial sum is dequantised by
 * its own activation and weight block scales,
 *   C[r,n] = sum_kb ( sum_{k in kb} A[r,k] B[e,n,k] ) * sa[r,kb] * sb[e,n/128,kb]
 * and activations are quantised per block with the per-token rule
 * (scale = max(amax_block, 1e-10)/448, code = e4m3(x / scale)).
 * ======================================================================== */

/* moe_permute_quant with block scales: scale_a [T*K, H/128] f32, row d
 * holding the scales of the token copied to row d. H % 128 == 0. Same
 * workspace as moe_permute_quant. Codes and scales bit-exact. */
MOE_API moe_status moe_permute_quant_block(const void* x, const int32_t* topk_ids,
                              int T, int H, int E, int K, void* a_q,
                              float* scale_a, int32_t* src2dst, int32_t* offsets,
                              void* ws, size_t ws_bytes, void* stream);

/* moe_grouped_gemm with block scales: scale_a [M, Kd/128] f32, scale_b
 * [E, N/128, Kd/128] f32; epilogues as moe_grouped_gemm (no row amax).
 * Kd % 128 == 0; N % 128 == 0 (SILU_MUL: N % 256 == 0, i.e. I % 128 == 0). */
MOE_API moe_status moe_grouped_gemm_block(const void* A, const float* scale_a,
                              const void* B, const float* scale_b,
                              const int32_t* offsets, int M, int N, int Kd, int E,
                              int epilogue, void* C, void* stream);

/* moe_act_quant with block scales: scale [M, I/128] f32. I % 128 == 0.
 * Bit-exact. */
MOE_API moe_status moe_act_quant_block(const void* h, int M, int I, void* q,
                              float* scale, void* stream);

/* Workspace bytes of moe_forward_block / moe_forward_block_host; with shared
 * experts pass E + n_shared and top_k + n_shared. 0 if H or I is not a
 * multiple of 128. */
MOE_API size_t moe_block_workspace_size(int T, int H, int I, int E, int K);

/* The whole layer in block FP8 (with n_shared shared experts as in
 * moe_forward_shared; 0 for none): s13 [E+n_shared, 2I/128, H/128],
 * s2 [E+n_shared, H/128, I/128]; otherwise as moe_forward_shared.
 * H % 128 == 0 and I % 128 == 0. */
MOE_API moe_status moe_forward_block(const void* x, const float* logits,
                              const float* bias, const void* w13,
                              const float* s13, const void* w2, const float* s2,
                              int T, int H, int I, int E, int n_shared,
                              int num_groups, int topk_group, int top_k,
                              int scoring, int renormalize,
                              float routed_scaling_factor, void* out, void* ws,
                              size_t ws_bytes, void* stream);

/* moe_forward_block with x, logits and out in host memory, as
 * moe_forward_host. */
MOE_API moe_status moe_forward_block_host(const void* x_host,
                              const float* logits_host, const float* bias,
                              const void* w13, const float* s13, const void* w2,
                              const float* s2, int T, int H, int I, int E,
                              int n_shared, int num_groups, int topk_group,
                              int top_k, int scoring, int renormalize,
                              float routed_scaling_factor, void* out_host,
                              void* ws, size_t ws_bytes, void* stream);

/* ==========================================================================
 * NVFP4: the FP4 format [P3] deploys DeepSeek-R1 in (modelopt_fp4; the
 * pages name it without writing it out). Reading, from NVIDIA's published
 * NVFP4 description: E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6),
 * one E4M3 scale per 16 consecutive elements along K, one fp32 global scale
 * per tensor; value = e2m1(q) * e4m3(s) * g. A 16-element block of x is
 * quantised with s = e4m3((amax / 6) / g) and q = e2m1(x / (e4m3(s) * g))
 * (IEEE fp32 divisions; nearest even, saturating; a block whose scale
 * decodes to 0 gets zero codes). The activations' global scales (ga1 for x,
 * ga2 for h) are inputs (calibrated input scales), as are the weights' g13[e]
 * and g2[e].
 * Packed layouts: codes two per byte along K, element 2j in the low nibble
 * of byte j; scales one byte per 16 elements:
 *   w13 [E,2I,H/2], s13 [E,2I,H/16], w2 [E,H,I/2], s2 [E,H,I/16] (bytes);
 *   g13, g2 [E] f32. H % 256 == 0 and I % 256 == 0.
 * The GEMMs take the weights' scales ARRANGED by moe_nvfp4_arrange_scales
 * (once, when the layer is set up): same bytes, in the order the kernel
 * copies them to tensor memory.
 * The GEMMs run on the block-scaled tensor-core MMA
 * (tcgen05.mma.kind::mxf4nvf4.block_scale, block 16, UE4M3 scales).
 * ======================================================================== */

/* moe_permute_quant in NVFP4 with global scale g > 0: a_q [T*K, H/2] packed
 * E2M1, sf [T*K, H/16] E4M3 block scales; src2dst, offsets and the workspace
 * as moe_permute_quant. Bit-exact. H % 16 == 0. */
MOE_API moe_status moe_permute_quant_nvfp4(const void* x, const int32_t* topk_ids, int T,
                                           int H, int E, int K, float g, void* a_q,
                                           uint8_t* sf, int32_t* src2dst, int32_t* offsets,
                                           void* ws, size_t ws_bytes, void* stream);

/* NVFP4 requantisation of h [M,I] bf16 with global scale g > 0:
 * q [M, I/2] packed E2M1, sf [M, I/16] E4M3. Bit-exact. I % 32 == 0. */
MOE_API moe_status moe_act_quant_nvfp4(const void* h, int M, int I, float g, void* q,
                                       uint8_t* sf, void* stream);

/*
 * moe_nvfp4_arrange_scales — the weights' block scales sb [E,N,Kd/16] (one
 * byte per 16 elements along K) rewritten into out (same size, a distinct
 * buffer) in the order moe_grouped_gemm_nvfp4 copies them to tensor memory:
 * for expert e, weight tile nb, K chunk c (256 elements) and MMA step j
 * (64 elements), 512 bytes holding at 16*(m%32) + 4*(m/32) + b scale 4j+b
 * of chunk c of the tile's row m. Tile rows: epilogue MOE_EPI_BF16, rows
 * 128*nb + m; MOE_EPI_SILU_MUL (w13, N = 2I), rows 64*nb + m for m < 64
 * (gate) and I + 64*nb + m - 64 (up). Kd % 256 == 0, N % 128 == 0.
 */
MOE_API moe_status moe_nvfp4_arrange_scales(const uint8_t* sb, int E, int N, int Kd,
                                            int epilogue, uint8_t* out, void* stream);

/* moe_grouped_gemm in NVFP4: A [M, Kd/2] packed, sfa [M, Kd/16], ga (the
 * activations' global scale); B [E, N, Kd/2] packed, sfb the weight scales
 * arranged by moe_nvfp4_arrange_scales for this epilogue, gb [E] f32;
 * acc[r,n] = sum_k a b sa sb (fp32), dequantised by ga * gb[e], then the
 * epilogue (no row amax). Kd % 256 == 0, N % 128 == 0. */
MOE_API moe_status moe_grouped_gemm_nvfp4(const void* A, const uint8_t* sfa, float ga,
                                          const void* B, const uint8_t* sfb, const float* gb,
                                          const int32_t* offsets, int M, int N, int Kd, int E,
                                          int epilogue, void* C, void* stream);

/*
 * moe_test_gemm_nvfp4_timeout — failure-detection test of the NVFP4 GEMM
 * pipelines (the pages have no counterpart), as moe_test_gemm_timeout:
 * runs moe_grouped_gemm_nvfp4 (whichever kernel its shapes select), except
 * that CTA 0 arms its pipeline stage number stall_stage (>= 0, counted over
 * its tiles) but never issues that stage's loads. Its bounded waits run out
 * (about 2 s), it sets MOE_DEV_PIPE_TIMEOUT, lets its issued copies and MMAs
 * land, frees its tensor memory and exits; the other CTAs finish. Returns
 * MOE_OK; moe_device_status then reports the timeout and the context stays
 * usable. C is left partly written. The same argument checks as
 * moe_grouped_gemm_nvfp4.
 */
MOE_API moe_status moe_test_gemm_nvfp4_timeout(const void* A, const uint8_t* sfa, float ga,
                                               const void* B, const uint8_t* sfb,
                                               const float* gb, const int32_t* offsets,
                                               int M, int N, int Kd, int E, int epilogue,
                                               void* C, int stall_stage, void* stream);

/* Workspace bytes of moe_forward_nvfp4 (with shared experts pass E+n_shared
 * and top_k+n_shared). */
MOE_API size_t moe_nvfp4_workspace_size(int T, int H, int I, int E, int K);

/* The whole layer in NVFP4: gate, pre-reorder + NVFP4 quant (ga1), w13 GEMM
 * + SiLU*mul, NVFP4 requant (ga2), w2 GEMM, weighted post-reorder; n_shared
 * shared experts as in moe_forward_shared (0 for none). Weights as above;
 * s13 and s2 arranged by moe_nvfp4_arrange_scales (s13 with
 * MOE_EPI_SILU_MUL, s2 with MOE_EPI_BF16); otherwise as moe_forward_shared. */
MOE_API moe_status moe_forward_nvfp4(const void* x, const float* logits, const float* bias,
                                     const void* w13, const uint8_t* s13, const float* g13,
                                     const void* w2, const uint8_t* s2, const float* g2,
                                     float ga1, float ga2, int T, int H, int I, int E,
                                     int n_shared, int num_groups, int topk_group, int top_k,
                                     int scoring, int renormalize,
                                     float routed_scaling_factor, void* out, void* ws,
                                     size_t ws_bytes, void* stream);

/* moe_forward_nvfp4 with x_host [T,H] bf16, logits_host [T,E] f32 and
 * out_host [T,H] bf16 in host memory, copied through the workspace on
 * `stream` (pinned memory keeps the copies asynchronous). */
MOE_API moe_status moe_forward_nvfp4_host(const void* x_host, const float* logits_host,
                                          const float* bias, const void* w13,
                                          const uint8_t* s13, const float* g13,
                                          const void* w2, const uint8_t* s2, const float* g2,
                                          float ga1, float ga2, int T, int H, int I, int E,
                                          int n_shared, int num_groups, int topk_group,
                                          int top_k, int scoring, int renormalize,
                                          float routed_scaling_factor, void* out_host,
                                          void* ws, size_t ws_bytes, void* stream);

/* ==========================================================================
 * Expert parallelism over R ranks: rank r holds experts [r*E/R, (r+1)*E/R)
 * (EPR = E/R of them) and its own tokens. [P3] Results deploys the layer
 * with --enable-ep-moe --ep-size 8 over 8 GPUs without describing the
 * exchange; it is read here as one all-to-all of token rows each way, done
 * by the caller (NCCL or any transport) between these calls:
 *   1. moe_gate, then moe_ep_dispatch on the rank's tokens: rows sorted by
 *      global expert, so rank r's rows are the block
 *      [offsets[r*EPR], offsets[(r+1)*EPR]) of a_q / scale_a;
 *      expert_counts[e] = offsets[e+1] - offsets[e].
 *   2. exchange: counts first (rank s sends expert_counts[r*EPR .. +EPR) to
 *      rank r, giving recv_counts [R][EPR]), then the rows and their scales
 *      (source blocks concatenated in source-rank order, Mr rows in all).
 *   3. moe_ep_expert_forward on the received rows with the local experts'
 *      weights: merge into expert-contiguous order (expert e: the rows of
 *      source 0, then source 1, ...), w13 GEMM + SiLU*mul, requant, w2 GEMM,
 *      then the output rows gathered back into arrival order (`back`).
 *   4. exchange back: each block of `back` returns to its source rank, in
 *      the order it came, so the rank's returned rows line up with its a_q.
 *   5. moe_ep_combine: the weighted top-k sum through src2dst (as
 *      moe_unpermute_sum).
 * With R = 1 and the exchanges as copies, the result is moe_forward's, bit
 * for bit. Every row's values are those of the one-GPU layer (the GEMMs and
 * the requant work per row).
 * ======================================================================== */

/* Scratch bytes of the merge table for R sources and EPR local experts. */
MOE_API size_t moe_ep_table_size(int R, int EPR);

/* moe_ep_dispatch — moe_permute_quant (same arguments, workspace and
 * outputs) plus expert_counts [E] i32 (out, device). E % R == 0 and
 * E <= 1024. */
MOE_API moe_status moe_ep_dispatch(const void* x, const int32_t* topk_ids, int T,
                              int H, int E, int K, int R, void* a_q,
                              float* scale_a, int32_t* src2dst, int32_t* offsets,
                              int32_t* expert_counts, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * moe_ep_recv_reorder — merge of the received rows into expert-contiguous
 * order. recv_rows [Mr,H] e4m3 and recv_scales [Mr] f32 in arrival order
 * (source blocks in source-rank order, each sorted by local expert);
 * recv_counts [R][EPR] i32 on the device (rows from source s for local
 * expert e; they must be >= 0 and sum to Mr, else MOE_DEV_BAD_OFFSETS is
 * raised, nothing is copied and the offsets are zero).
 * Out: a_q [Mr,H] e4m3 and scale_a [Mr] f32 in expert order, offsets
 * [EPR+1] i32, arrival2row [Mr] i32 (the expert-order row of each arrival
 * row). ws: moe_ep_table_size(R,EPR) bytes, 256-byte aligned.
 * Limits: H % 32 == 0, R*EPR <= 1024. Bit-exact (a permutation).
 */
MOE_API moe_status moe_ep_recv_reorder(const void* recv_rows, const float* recv_scales,
                              const int32_t* recv_counts, int R, int EPR, int Mr,
                              int H, void* a_q, float* scale_a, int32_t* offsets,
                              int32_t* arrival2row, void* ws, size_t ws_bytes,
                              void* stream);

/* moe_ep_return_gather — back[j,:] = down[arrival2row[j],:] for j < Mr
 * (bf16 rows of H values); an index outside [0,Mr) raises
 * MOE_DEV_BAD_OFFSETS and leaves that row unwritten. H % 8 == 0. */
MOE_API moe_status moe_ep_return_gather(const void* down, const int32_t* arrival2row,
                              int Mr, int H, void* back, void* stream);

/* Workspace bytes of moe_ep_expert_forward. */
MOE_API size_t moe_ep_expert_workspace_size(int Mr, int H, int I, int R, int EPR);

/*
 * moe_ep_expert_forward — the expert side of one step on this rank:
 * moe_ep_recv_reorder, moe_grouped_gemm (SILU_MUL) with w13 [EPR,2I,H] /
 * s13 [EPR,2I], moe_act_quant, moe_grouped_gemm (BF16) with w2 [EPR,H,I] /
 * s2 [EPR,H], moe_ep_return_gather into back [Mr,H] bf16, chained on one
 * stream. Arguments as those calls; ws: moe_ep_expert_workspace_size bytes,
 * 256-byte aligned. Limits: H % 32 == 0, I % 32 == 0, R*EPR <= 1024.
 */
MOE_API moe_status moe_ep_expert_forward(const void* recv_rows, const float* recv_scales,
                              const int32_t* recv_counts, int R, int EPR, int Mr,
                              int H, int I, const void* w13, const float* s13,
                              const void* w2, const float* s2, void* back,
                              void* ws, size_t ws_bytes, void* stream);

/* moe_ep_combine — the weighted top-k sum of the rows returned to this rank
 * (back_rows [T*K,H] bf16, in the order moe_ep_dispatch sorted them):
 * out[t,:] = bf16(sum_k topk_w[t,k] * back_rows[src2dst[t*K+k],:]), fp32 in
 * slot order, as moe_unpermute_sum. */
MOE_API moe_status moe_ep_combine(const void* back_rows, const int32_t* src2dst,
                              const float* topk_w, int T, int K, int H, void* out,
                              void* stream);

/* ---- pipelined host batches --------------------------------------------------
 * A serving loop feeds the layer batch after batch from host memory. Run one
 * call at a time, batch i+1's inputs cross the host link only after batch i's
 * output has come back, so the copies add to the compute. The pipelined entry
 * point below runs n batches through the same forward as moe_forward /
 * moe_forward_shared / moe_forward_block / moe_forward_nvfp4. Batch i+1's
 * inputs are copied in, and batch i-1's output copied out, while batch i
 * computes. Each batch's result is bit-identical to that batch run through
 * the matching device entry point alone.
 */
typedef enum {
  MOE_QUANT_TOKEN = 0, /* per-token FP8: moe_forward / moe_forward_shared */
  MOE_QUANT_BLOCK = 1, /* block-quantised FP8: moe_forward_block */
  MOE_QUANT_NVFP4 = 2  /* NVFP4: moe_forward_nvfp4 */
} moe_quant;

/* The layer a pipelined call runs: the arguments of the matching device
 * entry point, by name. s13 / s2 are f32 (token, block) or the arranged
 * E4M3 bytes of moe_nvfp4_arrange_scales (NVFP4); g13, g2, ga1 and ga2 are
 * read for NVFP4 only. Every pointer is a device pointer; the caller keeps
 * them valid while the call's work runs. */
typedef struct moe_layer {
  int quant; /* moe_quant */
  int T, H, I, E, n_shared, num_groups, topk_group, top_k, scoring, renormalize;
  float routed_scaling_factor;
  const float* bias;
  const void* w13;
  const void* s13;
  const void* w2;
  const void* s2;
  const float* g13;
  const float* g2;
  float ga1, ga2;
} moe_layer;

/* Workspace bytes moe_forward_host_pipelined needs for layer *L: the
 * matching forward's workspace plus two device slots for a batch's x,
 * logits and out. 0 if *L is invalid (NULL, an unknown quant or a size the
 * forward's workspace function rejects). */
MOE_API size_t moe_pipeline_workspace_size(const moe_layer* L);

/*
 * moe_forward_host_pipelined — n_batches forwards of layer *L over host
 * buffers: x_host[i] [T,H] bf16 and logits_host[i] [T,E] f32 in,
 * out_host[i] [T,H] bf16 out, for i = 0 .. n_batches-1.
 *
 * Streams. The forwards run on `stream`, in order. The copies into device
 * slot i % 2 and back out run on two internal copy streams of the current
 * device (created on first use and kept). Events order them:
 * - slot i % 2 is refilled only after batch i-2's forward has read it;
 * - batch i's forward waits for its inputs, and for batch i-2's output to
 *   have left the slot.
 * All of the call's work starts after the work already on `stream`, and
 * `stream` reaches the end of the call only once every output has landed.
 *
 * Host buffers. They must be pinned for the copies to overlap the compute
 * (pageable memory works, serialised) and stay valid until `stream` passes
 * the call. The same buffer may appear in several batches.
 *
 * Errors. MOE_ERR_INVALID_ARG for a NULL array or entry, n_batches < 1 or a
 * layer the forward rejects; MOE_ERR_WORKSPACE for a workspace below
 * moe_pipeline_workspace_size(L) or not 256-byte aligned. These are
 * returned before any work is queued. MOE_ERR_CUDA if a copy, event or
 * launch fails part way; earlier batches' work may then already be queued.
 */
MOE_API moe_status moe_forward_host_pipelined(const moe_layer* L, int n_batches,
                                              const void* const* x_host,
                                              const float* const* logits_host,
                                              void* const* out_host, void* ws,
                                              size_t ws_bytes, void* stream);

/*
 * moe_test_gemm_timeout — failure-detection test of the GEMM pipeline (the
 * pages have no counterpart). Runs moe_grouped_gemm, except that CTA 0 arms
 * its pipeline stage number stall_stage (>= 0, counted over its tiles) but
 * never issues that stage's loads. Its bounded waits then run out (about 2 s):
 * the CTA sets the device error word to MOE_DEV_PIPE_TIMEOUT, lets its
 * issued copies and MMAs land, frees its tensor memory and exits; the other
 * CTAs finish normally. The call itself returns MOE_OK; moe_device_status
 * then reports the timeout, and the context stays usable. C is left partly
 * written. The same argument checks as moe_grouped_gemm.
 */
MOE_API moe_status moe_test_gemm_timeout(const void* A, const float* scale_a,
                              const void* B, const float* scale_b,
                              const int32_t* offsets, int M, int N, int Kd,
                              int E, int epilogue, void* C, int stall_stage,
                              void* stream);

/*
 * moe_device_status — synchronises the current device, copies its device
 * error word into *code (one of MOE_DEV_*), clears it, and returns MOE_OK
 * when it was zero, MOE_ERR_DEVICE otherwise (MOE_ERR_CUDA if the copy
 * failed).
 */
MOE_API moe_status moe_device_status(int* code);

#ifdef __cplusplus
}
#endif
#endif
