// Bulk-copy (TMA, non-tensor) and mbarrier helpers, inline PTX for sm_100-
// family GPUs.  Every wait is bounded: after kSpinLimit failed polls the
// waiter raises the CTA's abort flag and reports DSV4KV_FAULT_TIMEOUT through
// the caller's fault counter, so a kernel can always return.  A producer
// waits (bounded again) for the copies it issued before its CTA exits; if
// that wait gives up too, a copy may still land in shared memory that a later
// CTA on the SM owns, so after a timeout fault every output of the launch --
// other CTAs' rows included -- is undefined.
#pragma once
#include <cstdint>

namespace dsv4kv {

// added to err_word when a wait gives up (never expected in normal operation)
constexpr int kFaultTimeout = 1 << 24;
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

// make the inits visible to the async proxy (the bulk copies' complete_tx)
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete.  Gives up (returns false) when
// *abort is raised by another thread, or after `limit` polls -- then it
// raises *abort itself and counts one timeout fault.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, int* err, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  if (atomicExch(const_cast<int*>(abort), 1) == 0 && err) atomicAdd(err, kFaultTimeout);
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err) {
  return mbar_wait_bounded(bar, parity, abort, err, kSpinLimit);
}

// Shared-memory accesses through generic pointers that the compiler cannot
// prove to be shared (e.g. inside a function that is not inlined).
__device__ __forceinline__ int ld_shared_s32(const int* p) {
  int v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ long long ld_shared_s64(const long long* p) {
  long long v;
  asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_s64(long long* p, long long v) {
  asm volatile("st.shared.b64 [%0], %1;" :: "r"(smem_u32(p)), "l"(v) : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization (launch_dependent) may start while the previous kernel in
// the stream is finishing; every thread waits in grid_dependency_wait before
// its first global memory access, so what the previous kernel wrote is
// complete and visible.  allow_dependent_launch lets the next such kernel
// start once every CTA of this one has called it or exited.  Both are no-ops
// in a normal launch.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 policy for data read exactly once
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy for data that every CTA of the grid reads
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// global -> shared bulk copy completing on `bar` (bytes: multiple of 16;
// both addresses 16-B aligned)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// shared -> global bulk copy in this thread's bulk group (bytes: multiple of
// 16; both addresses 16-B aligned)
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(dst), "r"(smem_u32(src)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// this thread's committed bulk stores have read their shared-memory source
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Named barriers over a subset of the CTA's warps (n: threads, a multiple of
// 32; every participating warp executes the instruction as a whole warp).
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(n) : "memory");
}

}  // namespace dsv4kv
