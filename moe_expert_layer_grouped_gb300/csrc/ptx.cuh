// Inline-PTX wrappers for the Blackwell (sm_103a) pieces of the grouped GEMM:
// mbarriers, TMA tensor loads, tensor-memory allocation, tcgen05.mma with
// shared-memory operand descriptors, tcgen05.commit and tcgen05.ld.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace moe {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up (returns
// false) once *abort is set or after `limit_ns` nanoseconds.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// ---- TMA ----------------------------------------------------------------------
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled load of box (x = innermost coordinate, y) into shared memory,
// completing on `bar` with the box's byte count.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x,
                                            int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 3-, 4- and 5-D tiled loads (coordinates fastest first), completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, int c3, int c4, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "l"(policy)
      : "memory");
}

// Four rows of a 2-D tensor (row coordinates r0..r3, any order, out-of-range
// rows read as the fill value) from column x, each row one box of the map
// (box one row high), landing as four consecutive box rows at dst;
// completing on `bar` with 4 x the box's bytes.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* m, uint64_t* bar, int x,
                                            int r0, int r1, int r2, int r3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "l"(policy)
      : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---- clusters -------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Shared::cluster address of the variable at local shared address `addr` in
// the CTA of the cluster with rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in a
// peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// 2-D tiled load into this CTA's shared memory for a CTA-pair MMA: the
// completion is counted on the mbarrier at `bar_cluster` (shared::cluster
// address), which may be in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx"
      "::bytes.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The 3-, 4- and 5-D loads for a CTA-pair MMA (completion counted on
// `bar_cluster`).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1, int c2,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx"
      "::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(void* dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1, int c2,
                                                 int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx"
      "::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d_pair(void* dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1, int c2,
                                                 int c3, int c4, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx"
      "::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "l"(policy)
      : "memory");
}

// tma_gather4 for a CTA-pair MMA (completion counted on `bar_cluster`, a
// shared::cluster address, possibly in the peer CTA).
__device__ __forceinline__ void tma_gather4_pair(void* dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int x, int r0, int r1,
                                                 int r2, int r3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4.mbarrier"
      "::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(
          smem_u32(dst)),
      "l"(m), "r"(bar_cluster), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "l"(policy)
      : "memory");
}

// ---- tensor memory / tcgen05 -------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warpgroup register reallocation: every warp of the warpgroup executes it.
// The increases of a CTA must be covered by its decreases and the registers
// it was launched with, else the increase waits.
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg range");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg range");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Tensor memory for a CTA pair: executed by one warp in each of the two CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (PTX ISA, tcgen05 "Shared Memory
// Descriptor") for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row (1024-byte) swizzle
// atoms stacked along M/N (stride byte offset 1024). The leading byte offset
// is unused for swizzled K-major layouts. Bits 46-47 hold the descriptor
// version (1) and bits 61-63 the layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4 (PTX ISA, tcgen05
// "Instruction descriptor" table for kind::f16 / f8f6f4): A and B e4m3, D fp32,
// both operands K-major, tile M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (0u << 7) | (0u << 10)           // A, B format: e4m3
         | (0u << 15) | (0u << 16)          // A, B K-major
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of tcgen05.mma.kind::mxf4nvf4.block_scale (PTX ISA,
// tcgen05 "Instruction descriptor" table for the block-scaled kinds): bits
// 4-5 B scale-factor id (0), 7-9 A type and 10-12 B type (E2M1 = 1), 15/16
// A/B K-major (0), 17-22 N >> 3, 23 scale type (0: UE4M3), 24-28 M >> 4,
// 29-30 A scale-factor id (0); D is fp32 for these kinds.
__host__ __device__ constexpr uint32_t idesc_nvfp4(int M, int N) {
  return (1u << 7) | (1u << 10)                // A, B: E2M1
         | ((uint32_t)(N >> 3) << 17)          // N / 8
         | ((uint32_t)(M >> 4) << 24);         // M / 16
}

// D[tmem] (+)= (A * SFA) (B * SFB)^T with E2M1 A/B in shared memory (two
// codes per byte, K-major, K = 64 per instruction) and one UE4M3 scale per
// 16 elements along K for every row of A and of B, read from tensor memory
// at sfa / sfb (.scale_vec::4X: four scales per row per instruction; PTX
// ISA, tcgen05 "Block Scaling" and its scale-factor layout in tensor
// memory: row m in lane m % 32, column m / 32 of the instruction's group).
__device__ __forceinline__ void mma_nvfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor (PTX ISA, tcgen05 "Shared Memory Descriptor",
// no-swizzle layout) of an unswizzled K-major block of 16-byte rows
// (8-row core matrices of 128 contiguous bytes, consecutive core matrices
// 128 bytes apart), the source of a tcgen05.cp of 32 rows x 128 bits.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;   // leading-dimension byte offset
  d |= (uint64_t)(128 >> 4) << 32;   // stride-dimension byte offset
  d |= (uint64_t)1 << 46;            // descriptor version
  return d;                           // layout bits 61-63: 0, no swizzle
}

// Copies 32 rows x 16 bytes from shared memory (descriptor sdesc) into
// tensor memory columns taddr .. taddr+3 of lanes 0..31, replicated into
// each of the four 32-lane quadrants (PTX ISA, tcgen05.cp: shape 32x128b
// with the .warpx4 multicast).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory writes before
// later async-proxy reads of them (tcgen05.cp, tcgen05.mma, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// CTA-pair MMA, issued by one thread of the even CTA: D (256 x N, rows
// 0..127 in this CTA's tensor memory, 128..255 in the peer's) (+)= A * B^T,
// A's rows 0..127 / 128..255 and B's rows 0..N/2-1 / N/2..N-1 read from this
// CTA's / the peer's shared memory at the same offsets.
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair version of the commit: arrive on the barrier at `bar`'s offset in
// every CTA of `cta_mask` once the pair's MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair_mcast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}


// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per
// thread). The registers are valid only after tmem_ld_wait() followed by
// reg_fence() on them.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (as the x32 form).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Writes r[0..15] of each lane into 16 consecutive TMEM columns from taddr,
// lane quadrant of the calling warp (lanes 32*(warp%4) ..); visible to later
// tcgen05 operations after tmem_st_wait() and a thread-sync fence.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Orders every later use of r after the preceding tmem_ld_wait().
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void reg_fence(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Loads 16 TMEM columns (32x32b.x16) into nxt, folds cur into acc
// (acc[i] += cur[i] * f, fp32 FMAs in pairs) while the load is in flight,
// then waits for the load. One asm statement, so nothing can read nxt
// before the wait; nxt is read-write so that it never shares a register
// with cur or acc.
__device__ __forceinline__ void tmem_ld_fold_x16(uint32_t taddr, uint32_t (&nxt)[16],
                                                const uint32_t (&cur)[16], float (&acc)[16],
                                                float f) {
  asm volatile(
      "{\n\t.reg .b64 fp, x, y;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%49];\n\t"
      "mov.b64 fp, {%48, %48};\n\t"
      "mov.b64 x, {%32, %33};\n\tmov.b64 y, {%16, %17};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%16, %17}, y;\n\t"
      "mov.b64 x, {%34, %35};\n\tmov.b64 y, {%18, %19};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%18, %19}, y;\n\t"
      "mov.b64 x, {%36, %37};\n\tmov.b64 y, {%20, %21};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%20, %21}, y;\n\t"
      "mov.b64 x, {%38, %39};\n\tmov.b64 y, {%22, %23};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%22, %23}, y;\n\t"
      "mov.b64 x, {%40, %41};\n\tmov.b64 y, {%24, %25};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%24, %25}, y;\n\t"
      "mov.b64 x, {%42, %43};\n\tmov.b64 y, {%26, %27};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%26, %27}, y;\n\t"
      "mov.b64 x, {%44, %45};\n\tmov.b64 y, {%28, %29};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%28, %29}, y;\n\t"
      "mov.b64 x, {%46, %47};\n\tmov.b64 y, {%30, %31};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%30, %31}, y;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t}"
      : "+r"(nxt[0]), "+r"(nxt[1]), "+r"(nxt[2]), "+r"(nxt[3]), "+r"(nxt[4]), "+r"(nxt[5]), "+r"(nxt[6]), "+r"(nxt[7]), "+r"(nxt[8]), "+r"(nxt[9]), "+r"(nxt[10]), "+r"(nxt[11]), "+r"(nxt[12]), "+r"(nxt[13]), "+r"(nxt[14]), "+r"(nxt[15]), "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]), "+f"(acc[6]), "+f"(acc[7]), "+f"(acc[8]), "+f"(acc[9]), "+f"(acc[10]), "+f"(acc[11]), "+f"(acc[12]), "+f"(acc[13]), "+f"(acc[14]), "+f"(acc[15])
      : "r"(cur[0]), "r"(cur[1]), "r"(cur[2]), "r"(cur[3]), "r"(cur[4]), "r"(cur[5]), "r"(cur[6]), "r"(cur[7]), "r"(cur[8]), "r"(cur[9]), "r"(cur[10]), "r"(cur[11]), "r"(cur[12]), "r"(cur[13]), "r"(cur[14]), "r"(cur[15]), "f"(f), "r"(taddr)
      : "memory");
}


__device__ __forceinline__ void tmem_ld_fold_x32(uint32_t taddr, uint32_t (&nxt)[32],
                                                const uint32_t (&cur)[32], float (&acc)[32],
                                                float f) {
  asm volatile(
      "{\n\t.reg .b64 fp, x, y;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%97];\n\t"
      "mov.b64 fp, {%96, %96};\n\t"
      "mov.b64 x, {%64, %65};\n\tmov.b64 y, {%32, %33};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%32, %33}, y;\n\t"
      "mov.b64 x, {%66, %67};\n\tmov.b64 y, {%34, %35};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%34, %35}, y;\n\t"
      "mov.b64 x, {%68, %69};\n\tmov.b64 y, {%36, %37};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%36, %37}, y;\n\t"
      "mov.b64 x, {%70, %71};\n\tmov.b64 y, {%38, %39};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%38, %39}, y;\n\t"
      "mov.b64 x, {%72, %73};\n\tmov.b64 y, {%40, %41};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%40, %41}, y;\n\t"
      "mov.b64 x, {%74, %75};\n\tmov.b64 y, {%42, %43};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%42, %43}, y;\n\t"
      "mov.b64 x, {%76, %77};\n\tmov.b64 y, {%44, %45};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%44, %45}, y;\n\t"
      "mov.b64 x, {%78, %79};\n\tmov.b64 y, {%46, %47};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%46, %47}, y;\n\t"
      "mov.b64 x, {%80, %81};\n\tmov.b64 y, {%48, %49};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%48, %49}, y;\n\t"
      "mov.b64 x, {%82, %83};\n\tmov.b64 y, {%50, %51};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%50, %51}, y;\n\t"
      "mov.b64 x, {%84, %85};\n\tmov.b64 y, {%52, %53};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%52, %53}, y;\n\t"
      "mov.b64 x, {%86, %87};\n\tmov.b64 y, {%54, %55};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%54, %55}, y;\n\t"
      "mov.b64 x, {%88, %89};\n\tmov.b64 y, {%56, %57};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%56, %57}, y;\n\t"
      "mov.b64 x, {%90, %91};\n\tmov.b64 y, {%58, %59};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%58, %59}, y;\n\t"
      "mov.b64 x, {%92, %93};\n\tmov.b64 y, {%60, %61};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%60, %61}, y;\n\t"
      "mov.b64 x, {%94, %95};\n\tmov.b64 y, {%62, %63};\n\t"
      "fma.rn.f32x2 y, x, fp, y;\n\tmov.b64 {%62, %63}, y;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t}"
      : "+r"(nxt[0]), "+r"(nxt[1]), "+r"(nxt[2]), "+r"(nxt[3]), "+r"(nxt[4]), "+r"(nxt[5]), "+r"(nxt[6]), "+r"(nxt[7]), "+r"(nxt[8]), "+r"(nxt[9]), "+r"(nxt[10]), "+r"(nxt[11]), "+r"(nxt[12]), "+r"(nxt[13]), "+r"(nxt[14]), "+r"(nxt[15]), "+r"(nxt[16]), "+r"(nxt[17]), "+r"(nxt[18]), "+r"(nxt[19]), "+r"(nxt[20]), "+r"(nxt[21]), "+r"(nxt[22]), "+r"(nxt[23]), "+r"(nxt[24]), "+r"(nxt[25]), "+r"(nxt[26]), "+r"(nxt[27]), "+r"(nxt[28]), "+r"(nxt[29]), "+r"(nxt[30]), "+r"(nxt[31]), "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]), "+f"(acc[6]), "+f"(acc[7]), "+f"(acc[8]), "+f"(acc[9]), "+f"(acc[10]), "+f"(acc[11]), "+f"(acc[12]), "+f"(acc[13]), "+f"(acc[14]), "+f"(acc[15]), "+f"(acc[16]), "+f"(acc[17]), "+f"(acc[18]), "+f"(acc[19]), "+f"(acc[20]), "+f"(acc[21]), "+f"(acc[22]), "+f"(acc[23]), "+f"(acc[24]), "+f"(acc[25]), "+f"(acc[26]), "+f"(acc[27]), "+f"(acc[28]), "+f"(acc[29]), "+f"(acc[30]), "+f"(acc[31])
      : "r"(cur[0]), "r"(cur[1]), "r"(cur[2]), "r"(cur[3]), "r"(cur[4]), "r"(cur[5]), "r"(cur[6]), "r"(cur[7]), "r"(cur[8]), "r"(cur[9]), "r"(cur[10]), "r"(cur[11]), "r"(cur[12]), "r"(cur[13]), "r"(cur[14]), "r"(cur[15]), "r"(cur[16]), "r"(cur[17]), "r"(cur[18]), "r"(cur[19]), "r"(cur[20]), "r"(cur[21]), "r"(cur[22]), "r"(cur[23]), "r"(cur[24]), "r"(cur[25]), "r"(cur[26]), "r"(cur[27]), "r"(cur[28]), "r"(cur[29]), "r"(cur[30]), "r"(cur[31]), "f"(f), "r"(taddr)
      : "memory");
}


// The x16 load and its wait in one statement: r is complete on return.
__device__ __forceinline__ void tmem_ld_sync_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// The x32 load and its wait in one statement: r is complete on return.
__device__ __forceinline__ void tmem_ld_sync_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_sync(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld_sync_x16(taddr, r);
}
__device__ __forceinline__ void tmem_ld_sync(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld_sync_x32(taddr, r);
}
__device__ __forceinline__ void tmem_ld_fold(uint32_t taddr, uint32_t (&nxt)[16],
                                             const uint32_t (&cur)[16], float (&acc)[16],
                                             float f) {
  tmem_ld_fold_x16(taddr, nxt, cur, acc, f);
}
__device__ __forceinline__ void tmem_ld_fold(uint32_t taddr, uint32_t (&nxt)[32],
                                             const uint32_t (&cur)[32], float (&acc)[32],
                                             float f) {
  tmem_ld_fold_x32(taddr, nxt, cur, acc, f);
}

// tmem_ld_32x32b_x16 / _x32 by the register count of the destination.
__device__ __forceinline__ void tmem_ld_32x32b(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld_32x32b_x16(taddr, r);
}
__device__ __forceinline__ void tmem_ld_32x32b(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld_32x32b_x32(taddr, r);
}

}  // namespace ptx
}  // namespace moe
