// mbarrier and bulk-copy (cp.async.bulk) helpers shared by the kernels that stage global
// memory in shared-memory rings, sm_103a.
#pragma once

#include <stdint.h>

#include "atom.cuh"

namespace coll {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async proxy and the other threads (follow
// with a CTA barrier).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// Bounded wait for the phase with the given parity: false once `limit` ns have passed or
// `stop()` (polled every 16 tries) returns true.
template <typename Stop>
__device__ __forceinline__ bool mbar_wait_until(uint64_t *bar, uint32_t parity, uint64_t limit,
                                                Stop stop) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u) {
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > limit) return false;
      if (stop()) return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit,
                                          const volatile uint32_t *abort_flag) {
  return mbar_wait_until(bar, parity, limit, [abort_flag]() { return *abort_flag != 0u; });
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to
// this CTA's shared memory; completion is counted on `bar`'s transaction count.
__device__ __forceinline__ void bulk_load(void *sdst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may
// start before the previous kernel in its stream has finished. griddep_wait() returns once
// that kernel has completed and its memory operations are visible; griddep_launch() lets the
// next kernel start as soon as every CTA of this grid has called it or exited.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Tensor copy of one 2-D box (the map's box size) at element coordinates (x, y) from global
// memory to this CTA's shared memory (128-byte aligned); completion is counted on `bar`'s
// transaction count. x times the element size must be a multiple of 16 bytes. A slot that
// threads read before is overwritten only after those reads have completed and the
// threads have synchronised with the issuing one (as with a consumer's release of a slot
// to a producer's copy).
__device__ __forceinline__ void tensor_load_2d(void *sdst, const void *tmap, uint32_t x,
                                               uint32_t y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(sdst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace coll
