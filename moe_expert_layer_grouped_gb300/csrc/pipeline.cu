// moe_forward_host_pipelined: batches from host memory through the layer with
// the host-link copies off the compute's critical path. The forwards run in
// order on the caller's stream. Batch i's inputs land in device slot i % 2
// from an internal H2D stream, and its output leaves slot i % 2 on an
// internal D2H stream. So while batch i computes, batch i+1's inputs come in
// and batch i-1's output goes out, on the GPU's copy engines. Events order
// the slots: a slot is refilled after the forward two batches back has read
// it, and a forward writes its output slot after the copy two batches back
// has drained it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "moe_gb300.h"

namespace {

constexpr size_t kAl = 256;
size_t al(size_t b) { return (b + kAl - 1) / kAl * kAl; }

// the matching forward's own workspace bytes (0: the layer is invalid)
size_t forward_ws(const moe_layer* L) {
  const int EA = L->E + L->n_shared, KA = L->top_k + L->n_shared;
  switch (L->quant) {
    case MOE_QUANT_TOKEN:
      return moe_workspace_size(L->T, L->H, L->I, EA, KA);
    case MOE_QUANT_BLOCK:
      return moe_block_workspace_size(L->T, L->H, L->I, EA, KA);
    case MOE_QUANT_NVFP4:
      return moe_nvfp4_workspace_size(L->T, L->H, L->I, EA, KA);
    default:
      return 0;
  }
}

struct Slots {
  size_t fws, x, l, o, total;  // offsets of slot 0; slot 1 follows each
};

Slots slots(const moe_layer* L) {
  Slots s{};
  s.fws = forward_ws(L);
  if (s.fws == 0 || L->T < 1) return s;
  const size_t xb = al((size_t)L->T * L->H * 2), lb = al((size_t)L->T * L->E * 4);
  size_t o = al(s.fws);
  s.x = o;
  o += 2 * xb;
  s.l = o;
  o += 2 * lb;
  s.o = o;
  o += 2 * xb;
  s.total = o;
  return s;
}

moe_status forward(const moe_layer* L, const void* x, const float* lg, void* out, void* ws,
                   size_t wsb, void* st) {
  switch (L->quant) {
    case MOE_QUANT_TOKEN:
      if (L->n_shared > 0)
        return moe_forward_shared(x, lg, L->bias, L->w13, static_cast<const float*>(L->s13),
                                  L->w2, static_cast<const float*>(L->s2), L->T, L->H, L->I,
                                  L->E, L->n_shared, L->num_groups, L->topk_group, L->top_k,
                                  L->scoring, L->renormalize, L->routed_scaling_factor, out, ws,
                                  wsb, st);
      return moe_forward(x, lg, L->bias, L->w13, static_cast<const float*>(L->s13), L->w2,
                         static_cast<const float*>(L->s2), L->T, L->H, L->I, L->E,
                         L->num_groups, L->topk_group, L->top_k, L->scoring, L->renormalize,
                         L->routed_scaling_factor, out, ws, wsb, st);
    case MOE_QUANT_BLOCK:
      return moe_forward_block(x, lg, L->bias, L->w13, static_cast<const float*>(L->s13), L->w2,
                               static_cast<const float*>(L->s2), L->T, L->H, L->I, L->E,
                               L->n_shared, L->num_groups, L->topk_group, L->top_k, L->scoring,
                               L->renormalize, L->routed_scaling_factor, out, ws, wsb, st);
    case MOE_QUANT_NVFP4:
      return moe_forward_nvfp4(x, lg, L->bias, L->w13, static_cast<const uint8_t*>(L->s13),
                               L->g13, L->w2, static_cast<const uint8_t*>(L->s2), L->g2, L->ga1,
                               L->ga2, L->T, L->H, L->I, L->E, L->n_shared, L->num_groups,
                               L->topk_group, L->top_k, L->scoring, L->renormalize,
                               L->routed_scaling_factor, out, ws, wsb, st);
    default:
      return MOE_ERR_INVALID_ARG;
  }
}

// the two copy streams of a device, created on first use and kept
bool copy_streams(cudaStream_t* h2d, cudaStream_t* d2h) {
  static std::mutex mu;
  static cudaStream_t in[64] = {}, out[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (in[dev] == nullptr) {
    cudaStream_t a = nullptr, b = nullptr;
    if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
      cudaStreamDestroy(a);
      return false;
    }
    in[dev] = a;
    out[dev] = b;
  }
  *h2d = in[dev];
  *d2h = out[dev];
  return true;
}

// the call's events, released when the call returns (an event still pending
// in a stream is released by the runtime once it completes)
struct Events {
  static constexpr int N = 7;  // start, in[2], used[2], out[2]
  cudaEvent_t e[N] = {};
  bool ok = true;
  Events() {
    for (auto& v : e)
      if (cudaEventCreateWithFlags(&v, cudaEventDisableTiming) != cudaSuccess) {
        v = nullptr;
        ok = false;
      }
  }
  ~Events() {
    for (auto v : e)
      if (v != nullptr) cudaEventDestroy(v);
  }
};

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace

extern "C" {

size_t moe_pipeline_workspace_size(const moe_layer* L) {
  if (L == nullptr) return 0;
  return slots(L).total;
}

moe_status moe_forward_host_pipelined(const moe_layer* L, int n_batches,
                                      const void* const* x_host,
                                      const float* const* logits_host, void* const* out_host,
                                      void* ws, size_t ws_bytes, void* stream) {
  if (L == nullptr || n_batches < 1 || x_host == nullptr || logits_host == nullptr ||
      out_host == nullptr)
    return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_batches; ++i)
    if (x_host[i] == nullptr || logits_host[i] == nullptr || out_host[i] == nullptr)
      return MOE_ERR_INVALID_ARG;
  const Slots S = slots(L);
  if (S.total == 0) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAl - 1)) != 0 || ws_bytes < S.total)
    return MOE_ERR_WORKSPACE;
  const size_t xb = (size_t)L->T * L->H * 2, lb = (size_t)L->T * L->E * 4;
  const size_t xs = al(xb), ls = al(lb);
  void* xd[2] = {at<void>(ws, S.x), at<void>(ws, S.x + xs)};
  float* ld[2] = {at<float>(ws, S.l), at<float>(ws, S.l + ls)};
  void* od[2] = {at<void>(ws, S.o), at<void>(ws, S.o + xs)};
  // the forward's own checks, once, on slot 0 before anything is queued
  // (T = 0 runs the checks only)
  {
    moe_layer probe = *L;
    probe.T = 0;
    const moe_status s = forward(&probe, xd[0], ld[0], od[0], ws, S.fws, stream);
    if (s != MOE_OK) return s;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStream_t h2d = nullptr, d2h = nullptr;
  if (!copy_streams(&h2d, &d2h)) return MOE_ERR_CUDA;
  Events ev;
  if (!ev.ok) return MOE_ERR_CUDA;
  cudaEvent_t start = ev.e[0], in[2] = {ev.e[1], ev.e[2]}, used[2] = {ev.e[3], ev.e[4]},
              out[2] = {ev.e[5], ev.e[6]};
  auto okc = [](cudaError_t e) { return e == cudaSuccess; };
  // everything after the work already on the caller's stream
  if (!okc(cudaEventRecord(start, cs)) || !okc(cudaStreamWaitEvent(h2d, start, 0)) ||
      !okc(cudaStreamWaitEvent(d2h, start, 0)))
    return MOE_ERR_CUDA;
  for (int i = 0; i < n_batches; ++i) {
    const int b = i & 1;
    // inputs into slot b once batch i-2's forward has read it
    if (i >= 2 && !okc(cudaStreamWaitEvent(h2d, used[b], 0))) return MOE_ERR_CUDA;
    if (!okc(cudaMemcpyAsync(xd[b], x_host[i], xb, cudaMemcpyHostToDevice, h2d)) ||
        !okc(cudaMemcpyAsync(ld[b], logits_host[i], lb, cudaMemcpyHostToDevice, h2d)) ||
        !okc(cudaEventRecord(in[b], h2d)))
      return MOE_ERR_CUDA;
    // the forward, once its inputs are in and batch i-2's output has left
    if (!okc(cudaStreamWaitEvent(cs, in[b], 0))) return MOE_ERR_CUDA;
    if (i >= 2 && !okc(cudaStreamWaitEvent(cs, out[b], 0))) return MOE_ERR_CUDA;
    const moe_status s = forward(L, xd[b], ld[b], od[b], ws, S.fws, stream);
    if (s != MOE_OK) return s;
    if (!okc(cudaEventRecord(used[b], cs))) return MOE_ERR_CUDA;
    // the output back to the host
    if (!okc(cudaStreamWaitEvent(d2h, used[b], 0)) ||
        !okc(cudaMemcpyAsync(out_host[i], od[b], xb, cudaMemcpyDeviceToHost, d2h)) ||
        !okc(cudaEventRecord(out[b], d2h)))
      return MOE_ERR_CUDA;
  }
  // the caller's stream passes the call once every output has landed
  for (int b = 0; b < (n_batches > 1 ? 2 : 1); ++b)
    if (!okc(cudaStreamWaitEvent(cs, out[b], 0))) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"
