// lt_async.cuh -- mbarriers and bulk (TMA) copies from global to shared memory,
// shared by the streamed top-k kernel and the compressor's ring.
//
// Waits are bounded: a wait makes at most a given number of try_wait calls,
// each suspending the thread for at most kSuspendNs, and reports whether the
// phase completed, so no kernel can spin forever on a copy.

#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lt {

constexpr uint32_t kWaitPolls = 1u << 16;  // try_wait calls before a wait gives up
constexpr uint32_t kSuspendNs = 20000;     // longest suspension per try_wait call

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also announces `bytes` of asynchronous transfers.
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Waits for the phase with the given parity to complete; the thread may be
// suspended for up to kSuspendNs per call instead of spinning.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs) : "memory");
  return ok != 0;
}
// Global -> this CTA's shared memory; completes `bytes` on the mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool ring_wait(uint64_t* bars, uint32_t ns, uint32_t seq, uint32_t polls) {
  uint64_t* bar = bars + (seq % ns);
  const uint32_t parity = (seq / ns) & 1u;
  for (uint32_t i = 0; i < polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

}  // namespace lt
