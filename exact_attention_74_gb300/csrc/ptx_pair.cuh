// ptx_pair.cuh -- primitives for two CTAs of a cluster that share tcgen05
// products (cta_group::2): the cluster rank and shared-memory address
// mapping, copies into and barrier arrivals on the other CTA's shared memory,
// cluster-scope bounded waits, and the pair forms of the tensor-memory
// allocation, the products and the commit.
//
// A kernel uses either these tcgen05 forms or the single-CTA ones of
// ptx.cuh, never both: the assembler rejects a function that mixes
// cta_group::1 and cta_group::2.
#pragma once

#include "ptx.cuh"

namespace fa {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The same shared-memory location in CTA `rank` of this cluster, as a
// shared::cluster address.
__device__ __forceinline__ uint32_t map_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t caddr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(caddr), "r"(v) : "memory");
}

// Copy `bytes` (a multiple of 16, both addresses 16-byte aligned) from this
// CTA's shared memory into another CTA's (dst from map_shared); completion
// is counted in bytes on the destination CTA's barrier `cbar` (map_shared).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t cbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "r"(src), "r"(bytes), "r"(cbar) : "memory");
}

// Arrive on a barrier in another CTA of the cluster (address from map_shared),
// releasing this thread's prior shared-memory writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cbar) : "memory");
}

// The same without release semantics, for hand-offs of tensor memory
// (ordered by the tcgen05 fences around the arrival) and of data that has
// already landed where the waiter's products read it.  A release at cluster
// scope costs about half a microsecond per arrival.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cbar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" :: "r"(cbar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait (cluster-scope acquire) for a CTA of a pair: on time-out it
// flags the status word and the abort flags of both CTAs, so that the other
// CTA stops waiting as well instead of running into its own time-out.
static __device__ __noinline__ bool pair_wait_slow(uint32_t bar, uint32_t parity, const DevCtl& ctl,
                                                   volatile int* abort, uint32_t peer_abort) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cl(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > ctl.timeout_ns) {
      atomicOr(ctl.status, kStatusTimeout);
      *abort = 1;
      st_cluster_u32(peer_abort, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, const DevCtl& ctl, volatile int* abort,
                                          uint32_t peer_abort) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  return pair_wait_slow(bar, parity, ctl, abort, peer_abort);
}

// Every thread of both CTAs; release / acquire at cluster scope.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tensor memory of a pair: one warp in each of the two CTAs executes the
// allocation (and later the release) together; both receive the same base.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}

// Arrive once on `bar` (the same offset) in each CTA of `cta_mask` when every
// pair product this thread issued so far has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(bar), "h"(cta_mask) : "memory");
}

// Pair product, issued by one thread of the even CTA: D (+)= A * B with M =
// 256 rows, rows [0, 128) in the even CTA's tensor memory and A rows from its
// shared memory (or tensor memory), rows [128, 256) likewise in the odd CTA;
// B's first N/2 columns come from the even CTA's shared memory and the rest
// from the odd CTA's, at the same descriptor address.
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
               : "memory");
}

__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
               : "memory");
}

// Shared-memory descriptor for an operand in 64-byte swizzled atoms (8 rows x
// 64 B, as TMA writes them with CU_TENSOR_MAP_SWIZZLE_64B): the same fields
// as sdesc_sw128 with layout code 4.  MN-major operand of 32 columns: sbo =
// 512 (next group of 8 K-rows); lbo would be the distance to the next
// 32-column atom and is unused at that width.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
         (1ull << 46) | (4ull << 61);
}

}  // namespace fa
