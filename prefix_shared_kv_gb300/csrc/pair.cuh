// Helpers for kernels whose tensor-core work runs on a pair of SMs (a cluster of two CTAs,
// tcgen05 .cta_group::2).  Every tcgen05 instruction of such a kernel uses .cta_group::2.
//
// The pair: CTA rank 0 (the even CTA) issues the MMAs.  With M = 256 each CTA holds 128 rows of A
// and its half of B's N columns in its own shared memory, at the same offsets in both CTAs, and
// receives its 128 rows of D (all N columns) in its own tensor memory at the same address.  A
// commit with a CTA mask arrives on the barrier at the same offset in every CTA of the mask.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace rx {
namespace pair {

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address in the shared memory of cluster CTA `rank` of the object at `saddr` in this CTA.
__device__ __forceinline__ uint32_t map_to(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// All threads of both CTAs; orders this CTA's earlier memory operations before the other CTA's
// later ones.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Arrival on a barrier of another CTA of the cluster (`caddr` from map_to).  Default semantics
// (release at CTA scope): what such an arrival publishes is tensor memory or shared memory that
// the pair's tensor core reads, ordered by the tcgen05 / proxy fences the caller issues before it.
// Release at cluster scope measured about twice the handoff latency of the whole pipeline.
__device__ __forceinline__ void arrive_remote(uint32_t caddr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// Phase test (default semantics: acquire at CTA scope), also for barriers whose arrivals come
// from the other CTA or from the pair's commits.
__device__ __forceinline__ bool try_wait_phase(uint32_t mbar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(mbar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// As tc::mbar_wait: gives up after `limit_ns` or once *abort is set;
// on giving up raises *abort, records RX_ERR_TIMEOUT in *status (first error wins), returns false.
__device__ __forceinline__ bool wait(uint32_t mbar, uint32_t parity, volatile int* abort,
                                     int32_t* status, uint64_t limit_ns) {
  if (try_wait_phase(mbar, parity, 0u)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (try_wait_phase(mbar, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort = 1;
      atomicCAS(status, 0, 5 /* RX_ERR_TIMEOUT */);
      return false;
    }
  }
}

// A progress counter in shared memory, published with release and read with acquire (CTA
// scope).  Plain loads and stores, not barrier operations: a thread that issues MMAs and commits
// can test it without being held until the tensor pipe has taken the MMAs before its commits,
// which every mbarrier operation after a commit is.
__device__ __forceinline__ void st_release(uint32_t saddr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(saddr) : "memory");
  return v;
}

// Tensor memory of the pair: one warp in each of the two CTAs runs these together.
__device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// D[tmem] (+)= A * B over the pair, A and B from shared-memory descriptors.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// The same with A from tensor memory (each CTA's 128 rows at a_tmem).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrives once on the barrier at offset `mbar` of every CTA in `cta_mask` when the MMAs this
// thread issued before it have completed.
__device__ __forceinline__ void commit_mc(uint32_t mbar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(mbar),
      "h"(cta_mask)
      : "memory");
}

}  // namespace pair
}  // namespace rx
