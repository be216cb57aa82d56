// qg_async.cuh -- mbarriers and bulk (TMA) copies into shared memory, shared
// by the tensor-core GEMM and the staged MoE down kernel.
//
// Every wait is bounded: a first try_wait with a suspend-time hint parks the
// warp until the phase completes; if it returns unready, a clock-bounded loop
// follows, which on timeout sets QG_DEV_ERR_WAIT in the kernel's device error
// word (read by qg_device_error) and lets the caller fall through.
#pragma once
#include <stdint.h>

#include "qgemm.h"

namespace qg {

constexpr long long ASYNC_WAIT_LIMIT = 4000000000LL;  // cycles (~2 s) before giving up
constexpr uint32_t ASYNC_SUSPEND_NS = 1000000;        // suspend-time hint of one try_wait (1 ms)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Arrive once per warp, from lane 0, without a divergent branch.
__device__ __forceinline__ void mbar_arrive_lane0(uint32_t bar, int lane) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %1, 0;\n\t"
      "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar), "r"(lane)
      : "memory");
}
// One try_wait on a phase: the warp may be parked until the phase completes
// (or the hint runs out), so a wait on a phase that is not complete yet costs
// no polling loop.
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ASYNC_SUSPEND_NS)
      : "memory");
  return ok;
}
// The rest of a wait whose first try failed: bounded by the clock (~2 s), after
// which QG_DEV_ERR_WAIT is set in *err and the caller falls through.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int32_t* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > ASYNC_WAIT_LIMIT) {
      atomicOr(err, QG_DEV_ERR_WAIT);
      return false;
    }
  }
  return true;
}
// Bounded wait on a phase of an mbarrier; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* err) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, err);
}
// As mbar_wait, with acquire semantics at cluster scope: the writes that other
// CTAs of the cluster made before their release arrivals on this barrier are
// visible once the phase has completed.
__device__ __forceinline__ uint32_t mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ASYNC_SUSPEND_NS)
      : "memory");
  return ok;
}
static __device__ __noinline__ bool mbar_wait_cluster_slow(uint32_t bar, uint32_t parity,
                                                           int32_t* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (clock64() - t0 > ASYNC_WAIT_LIMIT) {
      atomicOr(err, QG_DEV_ERR_WAIT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int32_t* err) {
  return mbar_try_wait_cluster(bar, parity) || mbar_wait_cluster_slow(bar, parity, err);
}
// Bulk copy of `bytes` contiguous bytes from global to this CTA's shared
// memory, completing on the mbarrier `bar` (its transaction count must have
// been raised by the bytes first). Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

}  // namespace qg
