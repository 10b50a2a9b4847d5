// CTA-pair (2-SM) tensor-core helpers: a cluster of two CTAs on two SMs runs one
// tcgen05.mma.cta_group::2 of M = 256, each CTA holding 128 rows of A and half of
// the N columns of B in its own shared memory, each CTA's tensor memory holding its
// 128 accumulator rows.  One thread of the even CTA (rank 0) issues the MMAs; the
// commits arrive on the barrier at the same offset in both CTAs; the odd CTA's
// producers and epilogue signal the even CTA's barriers through cluster addresses.
// Inline PTX only.
#pragma once

#include "tc.cuh"

namespace edge0 {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Cluster address of the shared-memory word at the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t cta_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
  return r;
}

// Every thread of both CTAs (hardware cluster barrier; used only where both CTAs
// are known to arrive: after set-up, before any early exit is possible).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM, pair-wide
// Collective over one warp of each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(slot)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem of both CTAs] (+)= A[256 rows: 128 per CTA] * B[N columns: N/2 per CTA]^T,
// kind::f16 (the instruction descriptor says bf16 or f16), issued by one thread of rank 0.
__device__ __forceinline__ void mma_pair_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive (once) on the barrier at `bar`'s offset in both CTAs when every pair MMA
// issued so far by this thread has completed.
__device__ __forceinline__ void mma_pair_commit_both(uint64_t* bar) {
  asm volatile(
      "{\n .reg .b16 m;\n mov.b16 m, 3;\n"
      " tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], m;\n}\n"
      ::"r"(smem_u32(bar)) : "memory");
}

// Arrive on rank 0's barrier only.
__device__ __forceinline__ void mma_pair_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------- barriers across the pair
// 2-D tile load into this CTA's shared memory, completion counted on a barrier of
// either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* tm, int x, int y, uint32_t bar_cl) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(tm), "r"(x), "r"(y), "r"(bar_cl) : "memory");
}

// Arrive with an expected byte count (no ordering of this thread's own accesses: the
// bytes come from bulk copies, whose completion the barrier counts).
__device__ __forceinline__ void mbar_arrive_expect_tx_cl(uint32_t bar_cl, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;"
               ::"r"(bar_cl), "r"(bytes) : "memory");
}

// Arrive on a barrier of either CTA of the pair with the default semantics (release
// at CTA scope): the pair's pipeline hand-offs, as between the CTAs of one cluster
// in general.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cl(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait (cluster-scope acquire) with the abort protocol of mbar_wait_abort.
__device__ __forceinline__ bool mbar_wait_cl_abort(uint64_t* bar, uint32_t parity, int* err, int* abort) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned int spins = 0;
  while (!mbar_try_wait_cl(bar, parity)) {
    if ((++spins & 63u) == 0) {
      if (abort && ld_relaxed_s32(abort)) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        if (err) atomicOr(err, kErrTimeout);
        if (abort) atomicExch(abort, 1);
        return false;
      }
    }
  }
  return true;
}

}  // namespace edge0
