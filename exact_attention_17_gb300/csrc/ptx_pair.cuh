// Inline-PTX wrappers for the two-SM kernel: cluster rank and barrier,
// shared::cluster addressing, remote mbarrier arrivals, cluster-scope waits
// and the cta_group::2 forms of the TMEM allocation, the MMA and the commit.
// Written from the PTX ISA's instruction descriptions; every wait is bounded.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace fa2dev {

// The two-SM form of the tensor-core instructions (cta_group::2) runs on a
// cluster of two CTAs: rank 0 (the leader) and rank 1 (its peer).

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster: release this thread's prior
// memory operations and wait until all threads of the cluster have arrived.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Shared::cluster address of the variable at `local` (a shared::cta
// address of this CTA) in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (in another
// CTA of the cluster), relaxed: no fence before the arrival.  A release at
// cluster scope fences all of the thread's memory operations across the
// cluster first, a membar of hundreds of cycles on the path the arrival
// sits on.  The callers arrive only once what the other CTA relies on is
// already complete: their own TMEM stores (after tcgen05.wait::st and
// tcgen05.fence::before_thread_sync), or copies they have seen land on
// their own barrier.
__device__ __forceinline__ void bar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// 32-bit store to a shared::cluster address.
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// try_wait with acquire semantics at cluster scope, for barriers that
// threads of another CTA arrive on.
__device__ __forceinline__ bool bar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// wait_bar at cluster scope (same bounds and result).
__device__ __forceinline__ bool wait_bar_cl(uint64_t* bar, uint32_t parity, volatile int* abort,
                                            uint64_t timeout_ns) {
  const uint32_t a = smem_addr(bar);
  if (bar_try_wait_cl(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (bar_try_wait_cl(a, parity)) return true;
    if ((it & 63u) == 0u) {
      if (abort != nullptr && *abort) return false;
      if (global_timer_ns() - t0 > timeout_ns) return false;
    }
  }
}

__device__ __forceinline__ bool bar_try_wait3_cl(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1,
                                                 uint32_t b2, uint32_t p2) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 q1, [%3], %4;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 q2, [%5], %6;\n\t"
      "and.pred q0, q0, q1;\n\t"
      "and.pred q0, q0, q2;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t}"
      : "=r"(ok)
      : "r"(b0), "r"(p0), "r"(b1), "r"(p1), "r"(b2), "r"(p2)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool wait_bar3_cl(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1,
                                             uint64_t* b2, uint32_t p2, volatile int* abort,
                                             uint64_t timeout_ns) {
  if (bar_try_wait3_cl(smem_addr(b0), p0, smem_addr(b1), p1, smem_addr(b2), p2)) return true;
  return wait_bar_cl(b0, p0, abort, timeout_ns) && wait_bar_cl(b1, p1, abort, timeout_ns) &&
         wait_bar_cl(b2, p2, abort, timeout_ns);
}

// TMEM allocation shared by a CTA pair: one warp of EACH of the two CTAs
// executes it; both receive the same column address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
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

// Two-SM MMA, issued by one thread of the leader CTA: D (+)= A * B^T with
// M = 256 rows, rows 0-127 from the leader (A from its shared memory, D in
// its TMEM) and rows 128-255 from the peer (same addresses there); each CTA
// holds half of B's N columns at the same shared-memory address.
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Two-SM MMA with A from TMEM (each CTA's own 128 rows).
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at `bar`'s offset in every CTA of `cta_mask`
// when every two-SM tensor-core operation this thread issued so far has
// completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(cta_mask)
      : "memory");
}

}  // namespace fa2dev
