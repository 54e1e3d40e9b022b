// Host-side launchers of the kernels, called by the C ABI (api.cu) after it
// has validated every argument. Each returns the CUDA error of its launch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Per-device state (device error word, SM count), set up on first use.
int* device_error_word();
int sm_count();

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// gate.cu: ids/w rows hold K + n_shared slots, the last n_shared being the
// shared experts E .. E+n_shared-1 with weight 1 (K + n_shared <= 32).
cudaError_t launch_gate(const float* logits, const float* bias, int T, int E, int G, int TG,
                        int K, int scoring, int renorm, float rsf, int32_t* ids, float* w,
                        int n_shared, cudaStream_t st);

// The launchers below take `pdl`: launch as a programmatic dependent of the
// previous kernel on the stream (the forward path chains its kernels this
// way; the single-step entry points launch plainly).

// permute.cu
size_t permute_ws_bytes(int T, int E);
// row_token non-null: a_q is [T, H], each token's codes stored once in token
// order, and row_token [T*K] receives the token of every permuted row (the
// grouped GEMM then gathers the rows, see launch_grouped_gemm).
cudaError_t launch_permute_quant(const void* x, const int32_t* ids, int T, int H, int E, int K,
                                 void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets,
                                 void* ws, int* err, cudaStream_t st, bool pdl = false,
                                 int32_t* row_token = nullptr);

// permute.cu: the same with one scale per 128 channels, scale_a [T*K, H/128]
// (H % 128 == 0).
cudaError_t launch_permute_quant_block(const void* x, const int32_t* ids, int T, int H, int E,
                                       int K, void* a_q, float* scale_a, int32_t* src2dst,
                                       int32_t* offsets, void* ws, int* err, cudaStream_t st,
                                       bool pdl = false);

// permute.cu: the same routing with NVFP4 quantisation (global scale g):
// a_q [T*K, H/2] (two E2M1 codes per byte), sf [T*K, H/16] E4M3 block scales.
cudaError_t launch_permute_quant_nvfp4(const void* x, const int32_t* ids, int T, int H, int E,
                                       int K, float g, void* a_q, uint8_t* sf, int32_t* src2dst,
                                       int32_t* offsets, void* ws, int* err, cudaStream_t st,
                                       bool pdl = false);

// permute.cu: device address of the fixed scratch used by
// moe_permute_quant_noalloc on the current device (nullptr on failure).
void* permute_static_scratch();

// gemm.cu
// Returns cudaErrorNotSupported when the TMA descriptors cannot be encoded.
// `early_table`: the offsets were written two or more kernels earlier on the
// stream, so the tile table is built before waiting for the previous kernel.
// row_token non-null: A is [T, Kd] in token order and permuted row r's
// tokens are row row_token[r] of it (loaded by four-row TMA gathers).
cudaError_t launch_grouped_gemm(const void* A, const float* scale_a, const void* B,
                                const float* scale_b, const int32_t* offsets, int M, int N,
                                int Kd, int E, int epilogue, void* C, float* row_amax, int* err,
                                cudaStream_t st, int stall_stage = -1, bool pdl = false,
                                bool early_table = false, const int32_t* row_token = nullptr,
                                int T = 0);
// Whether the grouped GEMM takes its many-rows-per-expert configuration.
bool gemm_many_rows(int M, int E);

// gemm_wide.cu: the per-token GEMM on CTA pairs with 256 weight rows per CTA
// (two accumulators), for many rows per expert and K of at least 32 blocks of
// 128 (SiLU: I % 256 == 0; bf16: N % 512 == 0). launch_grouped_gemm takes it
// by itself when it applies and no row amax, gather or stall test is asked.
bool gemm_wide_applies(int M, int N, int Kd, int E, int epilogue);
cudaError_t launch_grouped_gemm_wide(const void* A, const float* scale_a, const void* B,
                                     const float* scale_b, const int32_t* offsets, int M, int N,
                                     int Kd, int E, int epilogue, void* C, int* err,
                                     cudaStream_t st, bool pdl = false, bool early_table = false,
                                     int stall_stage = -1);

// gemm_block.cu: block scales, scale_a [M, Kd/128], scale_b [E, N/128, Kd/128]
// (N % 128 == 0, Kd % 128 == 0); no row amax.
cudaError_t launch_grouped_gemm_block(const void* A, const float* scale_a, const void* B,
                                      const float* scale_b, const int32_t* offsets, int M, int N,
                                      int Kd, int E, int epilogue, void* C, int* err,
                                      cudaStream_t st, bool pdl = false, bool early_table = false);

// act_quant.cu
cudaError_t launch_act_quant(const void* h, const float* row_amax, int M, int I, void* q,
                             float* scale, cudaStream_t st, bool pdl = false);

// act_quant.cu: one scale per 128 channels, scale [M, I/128] (I % 128 == 0).
cudaError_t launch_act_quant_block(const void* h, int M, int I, void* q, float* scale,
                                   cudaStream_t st, bool pdl = false);

// act_quant.cu: NVFP4 requantisation with global scale g: q [M, I/2],
// sf [M, I/16].
cudaError_t launch_act_quant_nvfp4(const void* h, int M, int I, float g, void* q, uint8_t* sf,
                                   cudaStream_t st, bool pdl = false);

// gemm_nvfp4.cu: NVFP4 grouped GEMM. A [M, Kd/2] and B [E, N, Kd/2] packed
// E2M1 (Kd % 256 == 0), sfa [M, Kd/16] E4M3 block scales, sfb the weights'
// scales arranged by launch_nvfp4_arrange_scales, ga and gb [E] fp32 global
// scales; acc * ga * gb[e] then the epilogue of launch_grouped_gemm (no row
// amax).
cudaError_t launch_nvfp4_arrange_scales(const uint8_t* sb, int E, int N, int Kd, int epilogue,
                                        uint8_t* out, cudaStream_t st);
cudaError_t launch_grouped_gemm_nvfp4(const void* A, const uint8_t* sfa, float ga, const void* B,
                                      const uint8_t* sfb, const float* gb,
                                      const int32_t* offsets, int M, int N, int Kd, int E,
                                      int epilogue, void* C, int* err, cudaStream_t st,
                                      bool pdl = false, bool early_table = false,
                                      int stall_stage = -1);

// gemm_nvfp4_wide.cu: the same GEMM with 256 weight rows per CTA, for many
// rows per expert (gemm_many_rows) when the weight rows split into 256-row
// tiles (SiLU: I % 128 == 0, bf16: N % 256 == 0); launch_grouped_gemm_nvfp4
// dispatches to it.
bool gemm_nvfp4_wide_applies(int M, int N, int Kd, int E, int epilogue);
cudaError_t launch_grouped_gemm_nvfp4_wide(const void* A, const uint8_t* sfa, float ga,
                                           const void* B, const uint8_t* sfb, const float* gb,
                                           const int32_t* offsets, int M, int N, int Kd, int E,
                                           int epilogue, void* C, int* err, cudaStream_t st,
                                           bool pdl, bool early_table, int stall_stage);

// unpermute.cu
cudaError_t launch_unpermute_sum(const void* down, const int32_t* src2dst, const float* w,
                                 int T, int K, int H, void* out, int* err, cudaStream_t st,
                                 bool pdl = false);

// ep.cu: expert-parallel merge of received rows and gather back.
// table: ep_table_bytes(R, EPR) bytes of scratch (256-byte aligned).
size_t ep_table_bytes(int R, int EPR);
int ep_max_table();  // largest R * EPR
cudaError_t launch_ep_counts(const int32_t* offsets, int E, int32_t* counts, cudaStream_t st,
                             bool pdl = false);
cudaError_t launch_ep_recv_reorder(const void* rows, const float* scales, const int32_t* cnt,
                                   int R, int EPR, int Mr, int H, void* a_q, float* scale_a,
                                   int32_t* offsets, int32_t* arrival2row, void* table,
                                   int* err, cudaStream_t st, bool pdl = false);
cudaError_t launch_ep_return_gather(const void* down, const int32_t* arrival2row, int Mr, int H,
                                    void* back, int* err, cudaStream_t st, bool pdl = false);

}  // namespace moe
