// Expert-parallel dispatch and combine: the steps on either side of the
// expert computation when the E experts are split over R ranks (E/R
// consecutive experts per rank), as in the pages' deployment with
// --enable-ep-moe --ep-size 8 ("[1/2] sgl-kernel: Fuse routed scaling factor
// into select_experts", sglang #8364, Results). The pages do not give the
// exchange itself; the reading here is an all-to-all of token rows each way:
//
//  dispatch (every rank, its own tokens): the pre-reorder of moe_permute_quant
//    sorts the (token, slot) pairs by GLOBAL expert, so the rows bound for
//    rank r are one contiguous block (experts [r*E/R, (r+1)*E/R)), already in
//    (local expert, token) order, with their FP8 codes and per-token scales;
//    the per-expert row counts (from the offsets) are exchanged first.
//  expert side (every rank, the rows it received): the received blocks, one
//    per source rank in rank order, are merged into expert-contiguous order
//    (expert e: source 0's rows, then source 1's, ...), the w13 GEMM, requant
//    and w2 GEMM run on the local experts, and the output rows are gathered
//    back into arrival order.
//  combine (every rank, its own tokens): the rows come back in the order they
//    were sent, so the weighted top-k sum indexes them through the same
//    src2dst as in the one-GPU layer.
//
// This file holds the merge (ep_table + ep_recv_copy) and the gather back
// (ep_return_gather); the exchange is the caller's (an all-to-all over NCCL
// or any transport); the other steps are the layer's own kernels.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTableThreads = 1024;

// One CTA. cnt [R][EPR]: rows received from source s for local expert e.
// Writes, in the workspace table:
//   off [EPR+1]          local expert offsets (expert-contiguous order)
//   arr [R*EPR]          arrival row of the first row of (s, e)
//   dst [R*EPR]          destination row of that row: off[e] + rows of e
//                        from sources before s
//   status [1]           0 ok; 1 the counts are negative or do not sum to Mr
// and the offsets to `offsets`.
__global__ void __launch_bounds__(kTableThreads)
    ep_table_kernel(const int32_t* __restrict__ cnt, int R, int EPR, int Mr,
                    int32_t* __restrict__ off, int32_t* __restrict__ arr,
                    int32_t* __restrict__ dst, int32_t* __restrict__ status,
                    int32_t* __restrict__ offsets, int* err) {
  chain_entry();
  __shared__ int wsum[kTableThreads / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = R * EPR;
  int bad = 0;
  // exclusive scan of the flattened counts (source-major): arrival starts
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += kTableThreads) {
    const int i = base + tid;
    const int v = i < n ? __ldg(cnt + i) : 0;
    bad |= v < 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = wsum[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += y;
      }
      wsum[lane] = wi - w;
    }
    __syncthreads();
    if (i < n) arr[i] = carry + wsum[warp] + incl - v;
    __syncthreads();
    if (tid == kTableThreads - 1) carry += wsum[warp] + incl;
    __syncthreads();
  }
  const int total = carry;
  // per local expert: the rows of all sources, then an exclusive scan over e
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < EPR; base += kTableThreads) {
    const int e = base + tid;
    int v = 0;
    if (e < EPR)
      for (int s = 0; s < R; ++s) v += __ldg(cnt + (int64_t)s * EPR + e);
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = wsum[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += y;
      }
      wsum[lane] = wi - w;
    }
    __syncthreads();
    if (e < EPR) {
      const int start = carry + wsum[warp] + incl - v;
      off[e] = start;
      int run = start;
      for (int s = 0; s < R; ++s) {
        dst[(int64_t)s * EPR + e] = run;
        run += __ldg(cnt + (int64_t)s * EPR + e);
      }
    }
    __syncthreads();
    if (tid == kTableThreads - 1) carry += wsum[warp] + incl;
    __syncthreads();
  }
  bad = __syncthreads_or(bad);
  if (tid == 0) {
    const int ok = !bad && total == Mr;
    off[EPR] = carry;
    status[0] = ok ? 0 : 1;
    if (!ok) flag_error(err, MOE_DEV_BAD_OFFSETS);
  }
  __syncthreads();
  // the offsets the GEMMs read: all zero when the counts are bad, so no
  // kernel after this one touches a row
  const int ok = !bad && total == Mr;
  for (int e = tid; e <= EPR; e += kTableThreads) offsets[e] = ok ? off[e] : 0;
}

constexpr int kCopyThreads = 256;
constexpr int kMaxTable = 1024;  // R * EPR entries held in shared memory

// Merge of the received rows into expert-contiguous order: one warp per
// arrival row j (grid-stride). (s, e) of row j is the last table entry whose
// arrival start is <= j; its destination is dst + (j - arr).
__global__ void __launch_bounds__(kCopyThreads)
    ep_recv_copy_kernel(const uint8_t* __restrict__ rows, const float* __restrict__ scales,
                        const int32_t* __restrict__ arr_g, const int32_t* __restrict__ dst_g,
                        const int32_t* __restrict__ status, int n, int Mr, int H,
                        uint8_t* __restrict__ a_q, float* __restrict__ scale_a,
                        int32_t* __restrict__ arrival2row) {
  chain_entry();
  __shared__ int arr[kMaxTable];
  __shared__ int dst[kMaxTable];
  if (__ldg(status) != 0) return;
  for (int i = threadIdx.x; i < n; i += kCopyThreads) {
    arr[i] = __ldg(arr_g + i);
    dst[i] = __ldg(dst_g + i);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int wpb = kCopyThreads / 32;
  const int nvec = H >> 4;  // 16-byte vectors per row
  for (int j = blockIdx.x * wpb + (threadIdx.x >> 5); j < Mr; j += gridDim.x * wpb) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (arr[mid] <= j) lo = mid;
      else hi = mid - 1;
    }
    const int d = dst[lo] + (j - arr[lo]);
    const uint4* src = reinterpret_cast<const uint4*>(rows + (int64_t)j * H);
    uint4* out = reinterpret_cast<uint4*>(a_q + (int64_t)d * H);
    for (int v = lane; v < nvec; v += 32) out[v] = __ldg(src + v);
    if (lane == 0) {
      scale_a[d] = __ldg(scales + j);
      arrival2row[j] = d;
    }
  }
}

// back[j, :] = down[arrival2row[j], :] (bf16 rows, 2H bytes): one warp per row.
__global__ void __launch_bounds__(kCopyThreads)
    ep_return_gather_kernel(const uint8_t* __restrict__ down,
                            const int32_t* __restrict__ arrival2row, int Mr, int H,
                            uint8_t* __restrict__ back, int* err) {
  chain_entry();
  const int lane = threadIdx.x & 31;
  const int wpb = kCopyThreads / 32;
  const int64_t rb = (int64_t)H * 2;
  const int nvec = (int)(rb >> 4);
  for (int j = blockIdx.x * wpb + (threadIdx.x >> 5); j < Mr; j += gridDim.x * wpb) {
    const int r = __ldg(arrival2row + j);
    if ((unsigned)r >= (unsigned)Mr) {
      if (lane == 0) flag_error(err, MOE_DEV_BAD_OFFSETS);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(down + (int64_t)r * rb);
    uint4* out = reinterpret_cast<uint4*>(back + (int64_t)j * rb);
    for (int v = lane; v < nvec; v += 32) out[v] = __ldg(src + v);
  }
}

__global__ void ep_counts_kernel(const int32_t* __restrict__ offsets, int E,
                                 int32_t* __restrict__ counts) {
  chain_entry();
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
    counts[e] = __ldg(offsets + e + 1) - __ldg(offsets + e);
}

int copy_grid(int rows) {
  const int wpb = kCopyThreads / 32;
  const int need = (rows + wpb - 1) / wpb;
  return std::max(1, std::min(need, sm_count() * 8));
}

}  // namespace

size_t ep_table_bytes(int R, int EPR) {
  return align_up((size_t)(EPR + 1) * 4) + 2 * align_up((size_t)R * EPR * 4) + align_up(4);
}

int ep_max_table() { return kMaxTable; }

cudaError_t launch_ep_counts(const int32_t* offsets, int E, int32_t* counts, cudaStream_t st,
                             bool pdl) {
  return launch_kernel(ep_counts_kernel, dim3((E + 255) / 256), dim3(256), 0, st, pdl, offsets,
                       E, counts);
}

cudaError_t launch_ep_recv_reorder(const void* rows, const float* scales, const int32_t* cnt,
                                   int R, int EPR, int Mr, int H, void* a_q, float* scale_a,
                                   int32_t* offsets, int32_t* arrival2row, void* table,
                                   int* err, cudaStream_t st, bool pdl) {
  char* t = static_cast<char*>(table);
  int32_t* off = reinterpret_cast<int32_t*>(t);
  t += align_up((size_t)(EPR + 1) * 4);
  int32_t* arr = reinterpret_cast<int32_t*>(t);
  t += align_up((size_t)R * EPR * 4);
  int32_t* dst = reinterpret_cast<int32_t*>(t);
  t += align_up((size_t)R * EPR * 4);
  int32_t* status = reinterpret_cast<int32_t*>(t);
  cudaError_t e = launch_kernel(ep_table_kernel, dim3(1), dim3(kTableThreads), 0, st, pdl, cnt,
                                R, EPR, Mr, off, arr, dst, status, offsets, err);
  if (e != cudaSuccess || Mr == 0) return e;
  return launch_kernel(ep_recv_copy_kernel, dim3(copy_grid(Mr)), dim3(kCopyThreads), 0, st, pdl,
                       static_cast<const uint8_t*>(rows), scales, (const int32_t*)arr,
                       (const int32_t*)dst, (const int32_t*)status, R * EPR, Mr, H,
                       static_cast<uint8_t*>(a_q), scale_a, arrival2row);
}

cudaError_t launch_ep_return_gather(const void* down, const int32_t* arrival2row, int Mr, int H,
                                    void* back, int* err, cudaStream_t st, bool pdl) {
  if (Mr == 0) return cudaSuccess;
  return launch_kernel(ep_return_gather_kernel, dim3(copy_grid(Mr)), dim3(kCopyThreads), 0, st,
                       pdl, static_cast<const uint8_t*>(down), arrival2row, Mr, H,
                       static_cast<uint8_t*>(back), err);
}

}  // namespace moe
