// C ABI of the MoE layer forward: argument validation, workspace layout and
// the one-stream orchestration of moe_forward. Declarations and the meaning
// of every argument are in include/moe_gb300.h.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

// The device error word: written by kernels that detect a fault, read and
// cleared by moe_device_status().
static __device__ int g_device_error;

int* device_error_word() {
  static std::mutex mu;
  static int* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

int sm_count() {
  static std::mutex mu;
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lk(mu);
  if (count[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    count[dev] = n > 0 ? n : 1;
  }
  return count[dev];
}

namespace {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxH = 16384;  // permute_quant keeps a row in registers

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return MOE_ERR_CUDA;
}

moe_status check_gate(const float* logits, const float* bias, int T, int E, int G, int TG,
                      int K, int scoring, const int32_t* ids, const float* w) {
  if (T < 0 || E < 1 || G < 1 || TG < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (E % G != 0 || TG > G || K > TG * (E / G)) return MOE_ERR_INVALID_ARG;
  if (scoring != MOE_SCORE_SIGMOID && scoring != MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || K > kMaxK || G > 64) return MOE_ERR_UNSUPPORTED;
  if (scoring == MOE_SCORE_SOFTMAX && (bias != nullptr || G != 1)) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!ok_ptr(logits) || !ok_ptr(ids) || !ok_ptr(w))) return MOE_ERR_INVALID_ARG;
  if (bias != nullptr && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Every check of a pre-reorder call except its workspace (shared by the
// workspace and the allocation-free entry points).
moe_status check_permute_args(const void* x, const int32_t* ids, int T, int H, int E, int K,
                              const void* a_q, const float* sa, const int32_t* s2d,
                              const int32_t* offsets) {
  if (T < 0 || H < 1 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (H % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || K > kMaxK || H > kMaxH) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * K >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(offsets)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ok_ptr(x) || !ok_ptr(ids) || !ok_ptr(a_q) || !ok_ptr(sa) || !ok_ptr(s2d)))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_permute(const void* x, const int32_t* ids, int T, int H, int E, int K,
                         const void* a_q, const float* sa, const int32_t* s2d,
                         const int32_t* offsets, const void* ws, size_t ws_bytes) {
  const moe_status s = check_permute_args(x, ids, T, H, E, K, a_q, sa, s2d, offsets);
  if (s != MOE_OK) return s;
  const size_t need = permute_ws_bytes(T, E);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 || ws_bytes < need)
    return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status check_gemm(const void* A, const float* sa, const void* B, const float* sb,
                      const int32_t* offsets, int M, int N, int Kd, int E, int epi,
                      const void* C, const float* row_amax) {
  if (M < 0 || N < 1 || Kd < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (epi != MOE_EPI_BF16 && epi != MOE_EPI_SILU_MUL) return MOE_ERR_INVALID_ARG;
  if (Kd % 32 != 0 || N % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (epi == MOE_EPI_SILU_MUL && N % 64 != 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= ((int64_t)1 << 31) || (int64_t)M >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(offsets) || !ok_ptr(B) || !ok_ptr(sb)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!ok_ptr(A) || !ok_ptr(sa) || !ok_ptr(C))) return MOE_ERR_INVALID_ARG;
  if (row_amax != nullptr && !aligned16(row_amax)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// moe_forward's workspace: every intermediate, 256-byte aligned pieces.
struct FwdLayout {
  size_t ids, w, perm, offsets, s2d, sa, sa2, a_q, h, q2, down, x_in, logits_in, out, total;
};

// block: 128-channel block scales (scale_a [M, H/128], scale_a2 [M, I/128]).
FwdLayout fwd_layout(int T, int H, int I, int E, int K, bool block = false) {
  FwdLayout L;
  const size_t M = (size_t)T * K;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes > 0 ? bytes : 1);
    return at;
  };
  L.ids = take(M * 4);
  L.w = take(M * 4);
  L.perm = take(permute_ws_bytes(T, E));
  L.offsets = take((size_t)(E + 1) * 4);
  L.s2d = take(M * 4);
  L.sa = take(M * 4 * (size_t)(block ? H / 128 : 1));
  L.sa2 = take(M * 4 * (size_t)(block ? I / 128 : 1));
  L.a_q = take(M * (size_t)H);
  L.h = take(M * (size_t)I * 2);
  L.q2 = take(M * (size_t)I);
  L.down = take(M * (size_t)H * 2);
  L.x_in = take((size_t)T * H * 2);
  L.logits_in = take((size_t)T * E * 4);
  L.out = take((size_t)T * H * 2);
  L.total = o;
  return L;
}

template <typename Tp>
Tp* at(void* ws, size_t off) {
  return reinterpret_cast<Tp*>(static_cast<char*>(ws) + off);
}

// S: shared experts, stored after the E routed ones (0 for moe_forward).
moe_status check_forward(const void* x, const float* logits, const float* bias, const void* w13,
                         const float* s13, const void* w2, const float* s2, int T, int H, int I,
                         int E, int S, int G, int TG, int K, int scoring, const void* out,
                         const void* ws, size_t ws_bytes, bool block) {
  if (S < 0) return MOE_ERR_INVALID_ARG;
  if (H < 1 || I < 1 || H % 32 != 0 || I % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (block && (H % 128 != 0 || I % 128 != 0)) return MOE_ERR_INVALID_ARG;
  if (H > kMaxH) return MOE_ERR_UNSUPPORTED;
  // the gate check without its output pointers (they live in the workspace)
  if (T < 0 || E < 1 || G < 1 || TG < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (E % G != 0 || TG > G || K > TG * (E / G)) return MOE_ERR_INVALID_ARG;
  if (scoring != MOE_SCORE_SIGMOID && scoring != MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
  if (E + S > kMaxE || K + S > kMaxK || G > 64) return MOE_ERR_UNSUPPORTED;
  if (scoring == MOE_SCORE_SOFTMAX && (bias != nullptr || G != 1)) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)(E + S) * 2 * I >= ((int64_t)1 << 31) ||
      (int64_t)(E + S) * H >= ((int64_t)1 << 31) || (int64_t)T * (K + S) >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(w13) || !ok_ptr(s13) || !ok_ptr(w2) || !ok_ptr(s2)) return MOE_ERR_INVALID_ARG;
  if (bias != nullptr && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ok_ptr(x) || !ok_ptr(logits) || !ok_ptr(out))) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 ||
      ws_bytes < fwd_layout(T, H, I, E + S, K + S, block).total)
    return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// The gate picks K of the E routed experts and appends the S shared ones
// (weight 1) to every token's row; from the permute on, the layer is a
// routed layer of E + S experts and K + S slots.
// block: the block-scaled FP8 steps (128-channel activation scales, 128 x 128
// weight scales) in place of the per-token ones.
moe_status run_forward(const void* x, const float* logits, const float* bias, const void* w13,
                       const float* s13, const void* w2, const float* s2, int T, int H, int I,
                       int E, int S, int G, int TG, int K, int scoring, int renorm, float rsf,
                       void* out, void* ws, cudaStream_t st, bool block) {
  const int EA = E + S, KA = K + S;  // experts and slots after the gate
  const FwdLayout L = fwd_layout(T, H, I, EA, KA, block);
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  const int M = T * KA;
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* s2d = at<int32_t>(ws, L.s2d);
  float* sa = at<float>(ws, L.sa);
  float* sa2 = at<float>(ws, L.sa2);
  void* a_q = at<void>(ws, L.a_q);
  void* h = at<void>(ws, L.h);
  void* q2 = at<void>(ws, L.q2);
  void* down = at<void>(ws, L.down);
  cudaError_t e;
  // The gate is launched plainly (after everything before it on the
  // stream); every later kernel of the step as a programmatic dependent of
  // the one before it.
  constexpr bool kChain = true;
  if ((e = launch_gate(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st)))
    return cuda_status(e);
  if (block) {
    if ((e = launch_permute_quant_block(x, ids, T, H, EA, KA, a_q, sa, s2d, offsets,
                                        at<void>(ws, L.perm), err, st, kChain)))
      return cuda_status(e);
    if ((e = launch_grouped_gemm_block(a_q, sa, w13, s13, offsets, M, 2 * I, H, EA,
                                       MOE_EPI_SILU_MUL, h, err, st, kChain)))
      return cuda_status(e);
    if ((e = launch_act_quant_block(h, M, I, q2, sa2, st, kChain))) return cuda_status(e);
    if ((e = launch_grouped_gemm_block(q2, sa2, w2, s2, offsets, M, H, I, EA, MOE_EPI_BF16,
                                       down, err, st, kChain, /*early_table=*/true)))
      return cuda_status(e);
  } else {
    // (the token-order rows of moe_permute_quant_rows with four-row TMA
    // gathers in the GEMM measured 2.5x slower for w13 than these K-fold
    // copies loaded as 64-row boxes, so the forward keeps the copies)
    if ((e = launch_permute_quant(x, ids, T, H, EA, KA, a_q, sa, s2d, offsets,
                                  at<void>(ws, L.perm), err, st, kChain)))
      return cuda_status(e);
    if ((e = launch_grouped_gemm(a_q, sa, w13, s13, offsets, M, 2 * I, H, EA, MOE_EPI_SILU_MUL,
                                 h, nullptr, err, st, -1, kChain)))
      return cuda_status(e);
    if ((e = launch_act_quant(h, nullptr, M, I, q2, sa2, st, kChain))) return cuda_status(e);
    if ((e = launch_grouped_gemm(q2, sa2, w2, s2, offsets, M, H, I, EA, MOE_EPI_BF16, down,
                                 nullptr, err, st, -1, kChain, /*early_table=*/true)))
      return cuda_status(e);
  }
  if ((e = launch_unpermute_sum(down, s2d, w, T, KA, H, out, err, st, kChain)))
    return cuda_status(e);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "unknown moe_status";
}

int moe_abi_version(void) { return (1 << 16) | 0; }

moe_status moe_gate(const float* logits, const float* bias, int T, int E, int num_groups,
                    int topk_group, int top_k, int scoring, int renormalize,
                    float routed_scaling_factor, int32_t* topk_ids, float* topk_w,
                    void* stream) {
  moe_status s = check_gate(logits, bias, T, E, num_groups, topk_group, top_k, scoring, topk_ids,
                            topk_w);
  if (s != MOE_OK) return s;
  return cuda_status(launch_gate(logits, bias, T, E, num_groups, topk_group, top_k, scoring,
                                 renormalize, routed_scaling_factor, topk_ids, topk_w, 0,
                                 static_cast<cudaStream_t>(stream)));
}

size_t moe_permute_workspace_size(int T, int E, int K) {
  (void)K;
  if (T < 0 || E < 1) return 0;
  return permute_ws_bytes(T, E);
}

moe_status moe_permute_quant(const void* x, const int32_t* topk_ids, int T, int H, int E, int K,
                             void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets,
                             void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_permute(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst, offsets, ws,
                               ws_bytes);
  if (s != MOE_OK) return s;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_permute_quant(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst,
                                          offsets, ws, err, static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute_quant_noalloc(const void* x, const int32_t* topk_ids, int T, int H,
                                     int E, int K, void* a_q, float* scale_a, int32_t* src2dst,
                                     int32_t* offsets, void* stream) {
  // the same checks as moe_permute_quant, with the fixed scratch as workspace;
  // all of them come before any CUDA call
  const moe_status s = check_permute_args(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst,
                                          offsets);
  if (s != MOE_OK) return s;
  if (permute_ws_bytes(T, E) > MOE_PERMUTE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* ws = permute_static_scratch();
  int* err = device_error_word();
  if (ws == nullptr || err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_permute_quant(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst,
                                          offsets, ws, err, static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gemm(const void* A, const float* scale_a, const void* B,
                            const float* scale_b, const int32_t* offsets, int M, int N, int Kd,
                            int E, int epilogue, void* C, float* row_amax, void* stream) {
  moe_status s = check_gemm(A, scale_a, B, scale_b, offsets, M, N, Kd, E, epilogue, C, row_amax);
  if (s != MOE_OK) return s;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_grouped_gemm(A, scale_a, B, scale_b, offsets, M, N, Kd, E, epilogue,
                                         C, row_amax, err, static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute_quant_rows(const void* x, const int32_t* topk_ids, int T, int H, int E,
                                  int K, void* a_tok, float* scale_a, int32_t* src2dst,
                                  int32_t* row_token, int32_t* offsets, void* ws,
                                  size_t ws_bytes, void* stream) {
  moe_status s = check_permute(x, topk_ids, T, H, E, K, a_tok, scale_a, src2dst, offsets, ws,
                               ws_bytes);
  if (s != MOE_OK) return s;
  if (T > 0 && !ok_ptr(row_token)) return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_permute_quant(x, topk_ids, T, H, E, K, a_tok, scale_a, src2dst,
                                          offsets, ws, err, static_cast<cudaStream_t>(stream),
                                          false, T > 0 ? row_token : nullptr));
}

moe_status moe_grouped_gemm_rows(const void* A_tok, int T, const int32_t* row_token,
                                 const float* scale_a, const void* B, const float* scale_b,
                                 const int32_t* offsets, int M, int N, int Kd, int E,
                                 int epilogue, void* C, float* row_amax, void* stream) {
  if (T < 0) return MOE_ERR_INVALID_ARG;
  moe_status s = check_gemm(A_tok, scale_a, B, scale_b, offsets, M, N, Kd, E, epilogue, C,
                            row_amax);
  if (s != MOE_OK) return s;
  if (M > 0 && (T < 1 || !ok_ptr(row_token))) return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_grouped_gemm(A_tok, scale_a, B, scale_b, offsets, M, N, Kd, E,
                                         epilogue, C, row_amax, err,
                                         static_cast<cudaStream_t>(stream), -1, false, false,
                                         row_token, T));
}

moe_status moe_test_gemm_timeout(const void* A, const float* scale_a, const void* B,
                                 const float* scale_b, const int32_t* offsets, int M, int N,
                                 int Kd, int E, int epilogue, void* C, int stall_stage,
                                 void* stream) {
  moe_status s = check_gemm(A, scale_a, B, scale_b, offsets, M, N, Kd, E, epilogue, C, nullptr);
  if (s != MOE_OK) return s;
  if (stall_stage < 0) return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_grouped_gemm(A, scale_a, B, scale_b, offsets, M, N, Kd, E, epilogue,
                                         C, nullptr, err, static_cast<cudaStream_t>(stream),
                                         stall_stage));
}

moe_status moe_act_quant(const void* h, const float* row_amax, int M, int I, void* q,
                         float* scale, void* stream) {
  if (M < 0 || I < 1 || I % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!ok_ptr(h) || !ok_ptr(q) || !ok_ptr(scale))) return MOE_ERR_INVALID_ARG;
  if (row_amax != nullptr && !aligned16(row_amax)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_act_quant(h, row_amax, M, I, q, scale,
                                      static_cast<cudaStream_t>(stream)));
}

moe_status moe_unpermute_sum(const void* down, const int32_t* src2dst, const float* topk_w,
                             int T, int K, int H, void* out, void* stream) {
  if (T < 0 || K < 1 || H < 1 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * K >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!ok_ptr(down) || !ok_ptr(src2dst) || !ok_ptr(topk_w) || !ok_ptr(out)))
    return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_unpermute_sum(down, src2dst, topk_w, T, K, H, out, err,
                                          static_cast<cudaStream_t>(stream)));
}

size_t moe_workspace_size(int T, int H, int I, int E, int K) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || K < 1) return 0;
  return fwd_layout(T, H, I, E, K).total;
}

}  // extern "C"

namespace moe {
namespace {

moe_status forward_device(const void* x, const float* logits, const float* bias, const void* w13,
                          const float* s13, const void* w2, const float* s2, int T, int H, int I,
                          int E, int S, int G, int TG, int K, int scoring, int renorm, float rsf,
                          void* out, void* ws, size_t ws_bytes, void* stream, bool block) {
  moe_status s = check_forward(x, logits, bias, w13, s13, w2, s2, T, H, I, E, S, G, TG, K,
                               scoring, out, ws, ws_bytes, block);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  return run_forward(x, logits, bias, w13, s13, w2, s2, T, H, I, E, S, G, TG, K, scoring, renorm,
                     rsf, out, ws, static_cast<cudaStream_t>(stream), block);
}

// The device address of a host buffer the GPU can read and write in place
// (pinned and mapped into the device's address space), else nullptr.
void* mapped_host_view(const void* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();  // not a CUDA-known pointer: clear the error
    return nullptr;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) return a.devicePointer;
  return nullptr;
}

// x, logits and out in host memory. When all three are pinned and mapped,
// the kernels read the inputs and write the output in host memory directly
// (the bytes still cross the host link inside the call); otherwise they are
// copied through the workspace on `stream`.
moe_status forward_host(const void* x_host, const float* logits_host, const float* bias,
                        const void* w13, const float* s13, const void* w2, const float* s2,
                        int T, int H, int I, int E, int S, int G, int TG, int K, int scoring,
                        int renorm, float rsf, void* out_host, void* ws, size_t ws_bytes,
                        void* stream, bool block) {
  if (T > 0 && (x_host == nullptr || logits_host == nullptr || out_host == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (S < 0 || H < 1 || I < 1 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (block && (H % 128 != 0 || I % 128 != 0)) return MOE_ERR_INVALID_ARG;
  if (T > 0) {
    void* xv = mapped_host_view(x_host);
    void* lv = mapped_host_view(logits_host);
    void* ov = mapped_host_view(out_host);
    if (xv != nullptr && lv != nullptr && ov != nullptr)
      return forward_device(xv, static_cast<const float*>(lv), bias, w13, s13, w2, s2, T, H, I,
                            E, S, G, TG, K, scoring, renorm, rsf, ov, ws, ws_bytes, stream,
                            block);
  }
  const FwdLayout L = fwd_layout(T < 0 ? 0 : T, H, I, E + S, K + S, block);
  void* x_d = at<void>(ws, L.x_in);
  float* l_d = at<float>(ws, L.logits_in);
  void* o_d = at<void>(ws, L.out);
  moe_status s = check_forward(x_d, l_d, bias, w13, s13, w2, s2, T, H, I, E, S, G, TG, K,
                               scoring, o_d, ws, ws_bytes, block);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * H * 2, lb = (size_t)T * E * 4;
  if (cudaMemcpyAsync(x_d, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(l_d, logits_host, lb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  s = run_forward(x_d, l_d, bias, w13, s13, w2, s2, T, H, I, E, S, G, TG, K, scoring, renorm,
                  rsf, o_d, ws, st, block);
  if (s != MOE_OK) return s;
  if (cudaMemcpyAsync(out_host, o_d, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_forward_shared(const void* x, const float* logits, const float* bias,
                              const void* w13, const float* s13, const void* w2, const float* s2,
                              int T, int H, int I, int E, int n_shared, int num_groups,
                              int topk_group, int top_k, int scoring, int renormalize,
                              float routed_scaling_factor, void* out, void* ws, size_t ws_bytes,
                              void* stream) {
  return forward_device(x, logits, bias, w13, s13, w2, s2, T, H, I, E, n_shared, num_groups,
                        topk_group, top_k, scoring, renormalize, routed_scaling_factor, out, ws,
                        ws_bytes, stream, false);
}

moe_status moe_forward(const void* x, const float* logits, const float* bias, const void* w13,
                       const float* s13, const void* w2, const float* s2, int T, int H, int I,
                       int E, int num_groups, int topk_group, int top_k, int scoring,
                       int renormalize, float routed_scaling_factor, void* out, void* ws,
                       size_t ws_bytes, void* stream) {
  return forward_device(x, logits, bias, w13, s13, w2, s2, T, H, I, E, 0, num_groups,
                        topk_group, top_k, scoring, renormalize, routed_scaling_factor, out, ws,
                        ws_bytes, stream, false);
}

moe_status moe_forward_shared_host(const void* x_host, const float* logits_host,
                                   const float* bias, const void* w13, const float* s13,
                                   const void* w2, const float* s2, int T, int H, int I, int E,
                                   int n_shared, int num_groups, int topk_group, int top_k,
                                   int scoring, int renormalize, float routed_scaling_factor,
                                   void* out_host, void* ws, size_t ws_bytes, void* stream) {
  return forward_host(x_host, logits_host, bias, w13, s13, w2, s2, T, H, I, E, n_shared,
                      num_groups, topk_group, top_k, scoring, renormalize,
                      routed_scaling_factor, out_host, ws, ws_bytes, stream, false);
}

moe_status moe_forward_host(const void* x_host, const float* logits_host, const float* bias,
                            const void* w13, const float* s13, const void* w2, const float* s2,
                            int T, int H, int I, int E, int num_groups, int topk_group,
                            int top_k, int scoring, int renormalize,
                            float routed_scaling_factor, void* out_host, void* ws,
                            size_t ws_bytes, void* stream) {
  return forward_host(x_host, logits_host, bias, w13, s13, w2, s2, T, H, I, E, 0, num_groups,
                      topk_group, top_k, scoring, renormalize, routed_scaling_factor, out_host,
                      ws, ws_bytes, stream, false);
}

// ---- block-quantised FP8 -------------------------------------------------------
moe_status moe_permute_quant_block(const void* x, const int32_t* topk_ids, int T, int H, int E,
                                   int K, void* a_q, float* scale_a, int32_t* src2dst,
                                   int32_t* offsets, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_permute(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst, offsets, ws,
                               ws_bytes);
  if (s != MOE_OK) return s;
  if (H % 128 != 0) return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_permute_quant_block(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst,
                                                offsets, ws, err,
                                                static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gemm_block(const void* A, const float* scale_a, const void* B,
                                  const float* scale_b, const int32_t* offsets, int M, int N,
                                  int Kd, int E, int epilogue, void* C, void* stream) {
  moe_status s = check_gemm(A, scale_a, B, scale_b, offsets, M, N, Kd, E, epilogue, C, nullptr);
  if (s != MOE_OK) return s;
  if (Kd % 128 != 0 || N % (epilogue == MOE_EPI_SILU_MUL ? 256 : 128) != 0)
    return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_grouped_gemm_block(A, scale_a, B, scale_b, offsets, M, N, Kd, E,
                                               epilogue, C, err,
                                               static_cast<cudaStream_t>(stream)));
}

moe_status moe_act_quant_block(const void* h, int M, int I, void* q, float* scale,
                               void* stream) {
  if (M < 0 || I < 1 || I % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!ok_ptr(h) || !ok_ptr(q) || !ok_ptr(scale))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_act_quant_block(h, M, I, q, scale, static_cast<cudaStream_t>(stream)));
}

size_t moe_block_workspace_size(int T, int H, int I, int E, int K) {
  if (T < 0 || H < 128 || I < 128 || E < 1 || K < 1 || H % 128 != 0 || I % 128 != 0) return 0;
  return fwd_layout(T, H, I, E, K, true).total;
}

moe_status moe_forward_block(const void* x, const float* logits, const float* bias,
                             const void* w13, const float* s13, const void* w2, const float* s2,
                             int T, int H, int I, int E, int n_shared, int num_groups,
                             int topk_group, int top_k, int scoring, int renormalize,
                             float routed_scaling_factor, void* out, void* ws, size_t ws_bytes,
                             void* stream) {
  return forward_device(x, logits, bias, w13, s13, w2, s2, T, H, I, E, n_shared, num_groups,
                        topk_group, top_k, scoring, renormalize, routed_scaling_factor, out, ws,
                        ws_bytes, stream, true);
}

moe_status moe_forward_block_host(const void* x_host, const float* logits_host,
                                  const float* bias, const void* w13, const float* s13,
                                  const void* w2, const float* s2, int T, int H, int I, int E,
                                  int n_shared, int num_groups, int topk_group, int top_k,
                                  int scoring, int renormalize, float routed_scaling_factor,
                                  void* out_host, void* ws, size_t ws_bytes, void* stream) {
  return forward_host(x_host, logits_host, bias, w13, s13, w2, s2, T, H, I, E, n_shared,
                      num_groups, topk_group, top_k, scoring, renormalize,
                      routed_scaling_factor, out_host, ws, ws_bytes, stream, true);
}

// ---- NVFP4 -----------------------------------------------------------------------
namespace {

bool nvfp4_dims_ok(int K) { return K >= 256 && K % 256 == 0; }

// moe_forward_nvfp4's workspace, 256-byte aligned pieces.
struct Fp4Layout {
  size_t ids, w, perm, offsets, s2d, a_q, sfa, h, q2, sfa2, down, x_in, logits_in, out, total;
};

Fp4Layout fp4_layout(int T, int H, int I, int E, int K) {
  Fp4Layout L;
  const size_t M = (size_t)T * K;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes > 0 ? bytes : 1);
    return at;
  };
  L.ids = take(M * 4);
  L.w = take(M * 4);
  L.perm = take(permute_ws_bytes(T, E));
  L.offsets = take((size_t)(E + 1) * 4);
  L.s2d = take(M * 4);
  L.a_q = take(M * (size_t)H / 2);
  L.sfa = take(M * (size_t)H / 16);
  L.h = take(M * (size_t)I * 2);
  L.q2 = take(M * (size_t)I / 2);
  L.sfa2 = take(M * (size_t)I / 16);
  L.down = take(M * (size_t)H * 2);
  L.x_in = take((size_t)T * H * 2);
  L.logits_in = take((size_t)T * E * 4);
  L.out = take((size_t)T * H * 2);
  L.total = o;
  return L;
}

moe_status check_gemm_nvfp4(const void* A, const void* sfa, float ga, const void* B,
                            const void* sfb, const float* gb, const int32_t* offsets, int M,
                            int N, int Kd, int E, int epi, const void* C) {
  if (M < 0 || N < 1 || Kd < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (epi != MOE_EPI_BF16 && epi != MOE_EPI_SILU_MUL) return MOE_ERR_INVALID_ARG;
  if (!nvfp4_dims_ok(Kd) || N % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (!(ga > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= ((int64_t)1 << 31) || (int64_t)M >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(offsets) || !ok_ptr(B) || !ok_ptr(sfb) || !ok_ptr(gb)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!ok_ptr(A) || !ok_ptr(sfa) || !ok_ptr(C))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status run_forward_nvfp4(const void* x, const float* logits, const float* bias,
                             const void* w13, const uint8_t* s13, const float* g13,
                             const void* w2, const uint8_t* s2, const float* g2, float ga1,
                             float ga2, int T, int H, int I, int E, int S, int G, int TG, int K,
                             int scoring, int renorm, float rsf, void* out, void* ws,
                             cudaStream_t st) {
  const int EA = E + S, KA = K + S;
  const Fp4Layout L = fp4_layout(T, H, I, EA, KA);
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  const int M = T * KA;
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* s2d = at<int32_t>(ws, L.s2d);
  void* a_q = at<void>(ws, L.a_q);
  uint8_t* sfa = at<uint8_t>(ws, L.sfa);
  void* h = at<void>(ws, L.h);
  void* q2 = at<void>(ws, L.q2);
  uint8_t* sfa2 = at<uint8_t>(ws, L.sfa2);
  void* down = at<void>(ws, L.down);
  cudaError_t e;
  constexpr bool kChain = true;
  if ((e = launch_gate(logits, bias, T, E, G, TG, K, scoring, renorm, rsf, ids, w, S, st)))
    return cuda_status(e);
  if ((e = launch_permute_quant_nvfp4(x, ids, T, H, EA, KA, ga1, a_q, sfa, s2d, offsets,
                                      at<void>(ws, L.perm), err, st, kChain)))
    return cuda_status(e);
  if ((e = launch_grouped_gemm_nvfp4(a_q, sfa, ga1, w13, s13, g13, offsets, M, 2 * I, H, EA,
                                     MOE_EPI_SILU_MUL, h, err, st, kChain)))
    return cuda_status(e);
  if ((e = launch_act_quant_nvfp4(h, M, I, ga2, q2, sfa2, st, kChain))) return cuda_status(e);
  if ((e = launch_grouped_gemm_nvfp4(q2, sfa2, ga2, w2, s2, g2, offsets, M, H, I, EA,
                                     MOE_EPI_BF16, down, err, st, kChain, /*early_table=*/true)))
    return cuda_status(e);
  if ((e = launch_unpermute_sum(down, s2d, w, T, KA, H, out, err, st, kChain)))
    return cuda_status(e);
  return MOE_OK;
}

}  // namespace

moe_status moe_permute_quant_nvfp4(const void* x, const int32_t* topk_ids, int T, int H, int E,
                                   int K, float g, void* a_q, uint8_t* sf, int32_t* src2dst,
                                   int32_t* offsets, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_permute(x, topk_ids, T, H, E, K, a_q, reinterpret_cast<const float*>(sf),
                               src2dst, offsets, ws, ws_bytes);
  if (s != MOE_OK) return s;
  if (H % 16 != 0 || !(g > 0.0f)) return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_permute_quant_nvfp4(x, topk_ids, T, H, E, K, g, a_q, sf, src2dst,
                                                offsets, ws, err,
                                                static_cast<cudaStream_t>(stream)));
}

moe_status moe_act_quant_nvfp4(const void* h, int M, int I, float g, void* q, uint8_t* sf,
                               void* stream) {
  if (M < 0 || I < 1 || I % 32 != 0 || !(g > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!ok_ptr(h) || !ok_ptr(q) || !ok_ptr(sf))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_act_quant_nvfp4(h, M, I, g, q, sf, static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gemm_nvfp4(const void* A, const uint8_t* sfa, float ga, const void* B,
                                  const uint8_t* sfb, const float* gb, const int32_t* offsets,
                                  int M, int N, int Kd, int E, int epilogue, void* C,
                                  void* stream) {
  moe_status s = check_gemm_nvfp4(A, sfa, ga, B, sfb, gb, offsets, M, N, Kd, E, epilogue, C);
  if (s != MOE_OK) return s;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_grouped_gemm_nvfp4(A, sfa, ga, B, sfb, gb, offsets, M, N, Kd, E,
                                               epilogue, C, err,
                                               static_cast<cudaStream_t>(stream)));
}

moe_status moe_test_gemm_nvfp4_timeout(const void* A, const uint8_t* sfa, float ga,
                                       const void* B, const uint8_t* sfb, const float* gb,
                                       const int32_t* offsets, int M, int N, int Kd, int E,
                                       int epilogue, void* C, int stall_stage, void* stream) {
  moe_status s = check_gemm_nvfp4(A, sfa, ga, B, sfb, gb, offsets, M, N, Kd, E, epilogue, C);
  if (s != MOE_OK) return s;
  if (stall_stage < 0) return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_grouped_gemm_nvfp4(A, sfa, ga, B, sfb, gb, offsets, M, N, Kd, E,
                                               epilogue, C, err,
                                               static_cast<cudaStream_t>(stream), false, false,
                                               stall_stage));
}

moe_status moe_forward_nvfp4_host(const void* x_host, const float* logits_host,
                                  const float* bias, const void* w13, const uint8_t* s13,
                                  const float* g13, const void* w2, const uint8_t* s2,
                                  const float* g2, float ga1, float ga2, int T, int H, int I,
                                  int E, int n_shared, int num_groups, int topk_group,
                                  int top_k, int scoring, int renormalize,
                                  float routed_scaling_factor, void* out_host, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (T > 0 && (x_host == nullptr || logits_host == nullptr || out_host == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (T < 0 || H < 1 || I < 1 || E < 1 || top_k < 1 || n_shared < 0) return MOE_ERR_INVALID_ARG;
  const Fp4Layout L = fp4_layout(T, H, I, E + n_shared, top_k + n_shared);
  void* x_d = at<void>(ws, L.x_in);
  float* l_d = at<float>(ws, L.logits_in);
  void* o_d = at<void>(ws, L.out);
  // the device entry point's checks, on the staging buffers
  moe_status s = moe_forward_nvfp4(x_d, l_d, bias, w13, s13, g13, w2, s2, g2, ga1, ga2, 0, H, I,
                                   E, n_shared, num_groups, topk_group, top_k, scoring,
                                   renormalize, routed_scaling_factor, o_d, ws, ws_bytes,
                                   stream);
  if (s != MOE_OK || T == 0) return s;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * H * 2, lb = (size_t)T * E * 4;
  if (cudaMemcpyAsync(x_d, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(l_d, logits_host, lb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  s = run_forward_nvfp4(x_d, l_d, bias, w13, s13, g13, w2, s2, g2, ga1, ga2, T, H, I, E,
                        n_shared, num_groups, topk_group, top_k, scoring, renormalize,
                        routed_scaling_factor, o_d, ws, st);
  if (s != MOE_OK) return s;
  if (cudaMemcpyAsync(out_host, o_d, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_nvfp4_arrange_scales(const uint8_t* sb, int E, int N, int Kd, int epilogue,
                                    uint8_t* out, void* stream) {
  if (E < 1 || N < 1 || !nvfp4_dims_ok(Kd) || N % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (epilogue != MOE_EPI_BF16 && epilogue != MOE_EPI_SILU_MUL) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(sb) || !ok_ptr(out) || sb == out) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_nvfp4_arrange_scales(sb, E, N, Kd, epilogue, out,
                                                 static_cast<cudaStream_t>(stream)));
}

size_t moe_nvfp4_workspace_size(int T, int H, int I, int E, int K) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || K < 1) return 0;
  return fp4_layout(T, H, I, E, K).total;
}

moe_status moe_forward_nvfp4(const void* x, const float* logits, const float* bias,
                             const void* w13, const uint8_t* s13, const float* g13,
                             const void* w2, const uint8_t* s2, const float* g2, float ga1,
                             float ga2, int T, int H, int I, int E, int n_shared,
                             int num_groups, int topk_group, int top_k, int scoring,
                             int renormalize, float routed_scaling_factor, void* out, void* ws,
                             size_t ws_bytes, void* stream) {
  if (!nvfp4_dims_ok(H) || !nvfp4_dims_ok(I)) return MOE_ERR_INVALID_ARG;
  if (!(ga1 > 0.0f) || !(ga2 > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(g13) || !ok_ptr(g2)) return MOE_ERR_INVALID_ARG;
  // the per-token layer's checks (shapes, gate, pointers), then this layer's
  // workspace
  moe_status s = check_forward(x, logits, bias, w13, reinterpret_cast<const float*>(s13), w2,
                               reinterpret_cast<const float*>(s2), T, H, I, E, n_shared,
                               num_groups, topk_group, top_k, scoring, out, ws, (size_t)-1,
                               false);
  if (s != MOE_OK) return s;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 ||
      ws_bytes < fp4_layout(T, H, I, E + n_shared, top_k + n_shared).total)
    return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  return run_forward_nvfp4(x, logits, bias, w13, s13, g13, w2, s2, g2, ga1, ga2, T, H, I, E,
                           n_shared, num_groups, topk_group, top_k, scoring, renormalize,
                           routed_scaling_factor, out, ws, static_cast<cudaStream_t>(stream));
}

// ---- expert-parallel dispatch / combine ---------------------------------------
size_t moe_ep_table_size(int R, int EPR) {
  if (R < 1 || EPR < 1) return 0;
  return ep_table_bytes(R, EPR);
}

moe_status moe_ep_dispatch(const void* x, const int32_t* topk_ids, int T, int H, int E, int K,
                           int R, void* a_q, float* scale_a, int32_t* src2dst, int32_t* offsets,
                           int32_t* expert_counts, void* ws, size_t ws_bytes, void* stream) {
  if (R < 1 || E < 1 || E % R != 0) return MOE_ERR_INVALID_ARG;
  if (R * (E / R) > ep_max_table() || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(expert_counts)) return MOE_ERR_INVALID_ARG;
  moe_status s = check_permute(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst, offsets, ws,
                               ws_bytes);
  if (s != MOE_OK) return s;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_permute_quant(x, topk_ids, T, H, E, K, a_q, scale_a, src2dst, offsets,
                                       ws, err, st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_ep_counts(offsets, E, expert_counts, st, true));
}

namespace {
moe_status check_ep_recv(const void* rows, const float* scales, const int32_t* cnt, int R,
                         int EPR, int Mr, int H) {
  if (R < 1 || EPR < 1 || Mr < 0 || H < 1 || H % 32 != 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)R * EPR > ep_max_table() || H > kMaxH) return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(cnt)) return MOE_ERR_INVALID_ARG;
  if (Mr > 0 && (!ok_ptr(rows) || !ok_ptr(scales))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Workspace of moe_ep_expert_forward: the merge table, then the local
// layer's intermediates, 256-byte aligned pieces.
struct EpLayout {
  size_t table, offsets, a_q, sa, a2r, h, q2, sa2, down, total;
};

EpLayout ep_layout(int Mr, int H, int I, int R, int EPR) {
  EpLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes > 0 ? bytes : 1);
    return at;
  };
  const size_t M = (size_t)(Mr > 0 ? Mr : 0);
  L.table = take(ep_table_bytes(R, EPR));
  L.offsets = take((size_t)(EPR + 1) * 4);
  L.a_q = take(M * H);
  L.sa = take(M * 4);
  L.a2r = take(M * 4);
  L.h = take(M * I * 2);
  L.q2 = take(M * I);
  L.sa2 = take(M * 4);
  L.down = take(M * H * 2);
  L.total = o;
  return L;
}
}  // namespace

moe_status moe_ep_recv_reorder(const void* recv_rows, const float* recv_scales,
                               const int32_t* recv_counts, int R, int EPR, int Mr, int H,
                               void* a_q, float* scale_a, int32_t* offsets,
                               int32_t* arrival2row, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_ep_recv(recv_rows, recv_scales, recv_counts, R, EPR, Mr, H);
  if (s != MOE_OK) return s;
  if (!ok_ptr(offsets)) return MOE_ERR_INVALID_ARG;
  if (Mr > 0 && (!ok_ptr(a_q) || !ok_ptr(scale_a) || !ok_ptr(arrival2row)))
    return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 ||
      ws_bytes < ep_table_bytes(R, EPR))
    return MOE_ERR_WORKSPACE;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_ep_recv_reorder(recv_rows, recv_scales, recv_counts, R, EPR, Mr, H,
                                            a_q, scale_a, offsets, arrival2row, ws, err,
                                            static_cast<cudaStream_t>(stream)));
}

moe_status moe_ep_return_gather(const void* down, const int32_t* arrival2row, int Mr, int H,
                                void* back, void* stream) {
  if (Mr < 0 || H < 1 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (Mr > 0 && (!ok_ptr(down) || !ok_ptr(arrival2row) || !ok_ptr(back)))
    return MOE_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  return cuda_status(launch_ep_return_gather(down, arrival2row, Mr, H, back, err,
                                             static_cast<cudaStream_t>(stream)));
}

size_t moe_ep_expert_workspace_size(int Mr, int H, int I, int R, int EPR) {
  if (Mr < 0 || H < 1 || I < 1 || R < 1 || EPR < 1) return 0;
  return ep_layout(Mr, H, I, R, EPR).total;
}

moe_status moe_ep_expert_forward(const void* recv_rows, const float* recv_scales,
                                 const int32_t* recv_counts, int R, int EPR, int Mr, int H,
                                 int I, const void* w13, const float* s13, const void* w2,
                                 const float* s2, void* back, void* ws, size_t ws_bytes,
                                 void* stream) {
  moe_status s = check_ep_recv(recv_rows, recv_scales, recv_counts, R, EPR, Mr, H);
  if (s != MOE_OK) return s;
  if (I < 1 || I % 32 != 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)EPR * 2 * I >= ((int64_t)1 << 31) || (int64_t)EPR * H >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(w13) || !ok_ptr(s13) || !ok_ptr(w2) || !ok_ptr(s2)) return MOE_ERR_INVALID_ARG;
  if (Mr > 0 && !ok_ptr(back)) return MOE_ERR_INVALID_ARG;
  const EpLayout L = ep_layout(Mr, H, I, R, EPR);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 ||
      ws_bytes < L.total)
    return MOE_ERR_WORKSPACE;
  int* err = device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  void* a_q = at<void>(ws, L.a_q);
  float* sa = at<float>(ws, L.sa);
  int32_t* a2r = at<int32_t>(ws, L.a2r);
  void* h = at<void>(ws, L.h);
  void* q2 = at<void>(ws, L.q2);
  float* sa2 = at<float>(ws, L.sa2);
  void* down = at<void>(ws, L.down);
  // merge -> w13 GEMM + SiLU*mul -> requant -> w2 GEMM -> back to arrival
  // order, each a programmatic dependent of the one before (the merge table
  // first, launched plainly)
  cudaError_t e;
  if ((e = launch_ep_recv_reorder(recv_rows, recv_scales, recv_counts, R, EPR, Mr, H, a_q, sa,
                                  offsets, a2r, at<void>(ws, L.table), err, st, false)))
    return cuda_status(e);
  if (Mr == 0) return MOE_OK;
  if ((e = launch_grouped_gemm(a_q, sa, w13, s13, offsets, Mr, 2 * I, H, EPR, MOE_EPI_SILU_MUL,
                               h, nullptr, err, st, -1, true)))
    return cuda_status(e);
  if ((e = launch_act_quant(h, nullptr, Mr, I, q2, sa2, st, true))) return cuda_status(e);
  if ((e = launch_grouped_gemm(q2, sa2, w2, s2, offsets, Mr, H, I, EPR, MOE_EPI_BF16, down,
                               nullptr, err, st, -1, true, /*early_table=*/true)))
    return cuda_status(e);
  return cuda_status(launch_ep_return_gather(down, a2r, Mr, H, back, err, st, true));
}

moe_status moe_ep_combine(const void* back_rows, const int32_t* src2dst, const float* topk_w,
                          int T, int K, int H, void* out, void* stream) {
  return moe_unpermute_sum(back_rows, src2dst, topk_w, T, K, H, out, stream);
}

moe_status moe_device_status(int* code) {
  if (code == nullptr) return MOE_ERR_INVALID_ARG;
  *code = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  return v == 0 ? MOE_OK : MOE_ERR_DEVICE;
}

}  // extern "C"
