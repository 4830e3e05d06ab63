// ptx_pair.cuh -- inline-PTX pieces for kernels whose tensor-core products
// span a pair of CTAs (tcgen05 .cta_group::2): a cluster of two CTAs on two
// SMs, where the even-ranked CTA issues M = 256 products whose A rows are
// split between the two CTAs' shared memory (128 rows each, same offset)
// and whose B columns are split the same way (N/2 each, the lower half in
// the even CTA), and each CTA's tensor memory receives its own 128 rows of
// the result.
//
// Every tcgen05 instruction of such a kernel carries .cta_group::2, the
// tensor-memory allocation included, which both CTAs perform (one warp
// each) and which yields the same columns in both.
#pragma once

#include "ptx.cuh"

namespace mha {

template <uint32_t kCols>
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_slot_smem) {
  static_assert(kCols >= 32 && kCols <= 512 && (kCols & (kCols - 1)) == 0, "TMEM columns");
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_slot_smem),
               "r"(kCols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <uint32_t kCols>
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kCols)
               : "memory");
}

// D[tmem, both CTAs] (+)= A[smem desc, 128 rows per CTA] * B[smem desc,
// N/2 columns per CTA]^T, issued by the even CTA only.
__device__ __forceinline__ void umma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrive once on the mbarrier at offset `bar` in every CTA of `cta_mask`
// when the pair's tcgen05 operations issued so far by this thread have
// completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask));
}

// The same, arriving on this CTA's own barrier only.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar));
}

// Tiled loads into this CTA's shared memory whose completion (transaction
// bytes) is signalled on `cbar`, a shared::cluster address that may name the
// peer CTA's barrier (from mapa).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cbar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cbar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cbar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cbar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// mbar_wait for a barrier of this CTA that the peer CTA arrives on: the
// acquire is at cluster scope, pairing with mbar_arrive_cluster's release.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  const WaitCtl& ctl) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*ctl.abort_flag) return false;
      if (global_timer_ns() - t0 > ctl.limit_ns) {
        *ctl.abort_flag = 1;
        atomicOr(ctl.err, kErrTimeout);
        return false;
      }
    }
  }
}

// Arrive on an mbarrier named by a shared::cluster address (this CTA's or
// the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar)
               : "memory");
}

}  // namespace mha
