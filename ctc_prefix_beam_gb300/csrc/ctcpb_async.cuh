// Bulk asynchronous copies into shared memory that complete on an mbarrier,
// with bounded waits (a wait that runs out reports failure instead of hanging).
#pragma once

#include "ctcpb_internal.cuh"

namespace ctcpb {

constexpr long long kWaitSpins = 1ll << 18;  // bounded mbarrier wait (each try sleeps <= 2 us)
constexpr int kExitWaits = 8;  // further bounded waits for a copy in flight before a warp exits on a timeout

__device__ __forceinline__ unsigned saddr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(u64* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(saddr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(u64* bar, unsigned bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(saddr(bar)),
      "r"(bytes)
      : "memory");
}
// bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// into shared memory, completing on the barrier
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, u64* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(saddr(dst)),
      "l"(src), "r"(bytes), "r"(saddr(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_test(u64* bar, unsigned parity) {
  unsigned ok;
  // the suspend hint lets the warp sleep in the barrier until the copy lands
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 2000;\n selp.u32 %0, 1, 0, "
      "p;\n}\n"
      : "=r"(ok)
      : "r"(saddr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait for a phase of a barrier; false if it gave up
__device__ __forceinline__ bool mbar_wait(u64* bar, unsigned parity) {
  for (long long i = 0; i < kWaitSpins; ++i) {
    if (mbar_test(bar, parity)) return true;
  }
  return false;
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// order this thread's earlier generic-proxy accesses of shared memory before
// its later bulk copies into it
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// Asynchronous copies global -> shared of 4 or 16 bytes (16: both addresses
// 16-byte aligned); they complete at cp_wait_all, and a barrier after it makes
// them visible to the other threads.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(saddr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// release store / acquire load of a flag in global memory (device scope)
__device__ __forceinline__ void st_release_u32(u32* p, u32 v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ u32 ld_acquire_u32(const u32* p) {
  u32 v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// order generic-proxy accesses of global memory (made visible by an acquire)
// before this thread's later bulk copies that read it
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

}  // namespace ctcpb
