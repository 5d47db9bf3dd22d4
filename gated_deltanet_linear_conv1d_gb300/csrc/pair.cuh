// pair.cuh - clusters and CTA pairs for libgdn's GEMM kernels: the 2-SM
// tcgen05 MMA (cta_group::2), in which the even CTA of a pair issues MMAs of
// M = 256 whose A rows come 128 from each CTA's shared memory, whose B rows
// come half from each, and whose accumulator rows land 128 in each CTA's tensor
// memory; plus the cluster-scope barriers and addresses that go with it.
#pragma once

#include <stdint.h>

#include "device.cuh"

namespace gdn {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster; orders the memory accesses before it
// (release) against those after it (acquire) at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  return a;
}

// One arrival on a barrier given by its shared::cluster address (possibly another
// CTA's), with release semantics at CTA scope only. The callers hand back a
// tensor-memory buffer whose tcgen05.ld reads have completed (tcgen05.wait::ld,
// then tcgen05.fence::before_thread_sync); no memory written before the arrival
// is read after it. A cluster-scope release would be a fence that also waits
// for every global store this thread still has in flight (the epilogue's): in
// the FP8 pair kernel, which arrives once per K block, that fence halved the rate.
__device__ __forceinline__ void arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// `bar_cluster`, a barrier of the pair (a shared::cluster address, here the even
// CTA's), with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* tmap, int x, int y, uint32_t bar_cluster,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}

// Tensor memory for the pair: one warp of each CTA executes these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrives once on `bar` in the CTAs of `mask` (the pair) when the pair's MMAs
// issued so far by this thread have completed.
__device__ __forceinline__ void commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                   "r"(smem_u32(bar)), "h"(mask)
               : "memory");
}

// One MMA of the pair, issued by the even CTA: D (this CTA's and the partner's
// tensor memory at the same address, 128 rows each) (+)= A (128 rows from each
// CTA's shared memory at the descriptor's address) B^T (N / 2 rows from each).
// kF8: kind::f8f6f4 (E4M3 operands, K = 32 per MMA); else kind::f16 (bf16, K = 16).
template <bool kF8>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  if constexpr (kF8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

}  // namespace gdn
