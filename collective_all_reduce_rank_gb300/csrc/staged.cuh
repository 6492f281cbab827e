// staged.cuh -- pieces shared by the kernels that stage messages in shared
// memory with bulk copies and hand them between warps with mbarriers (the
// staged ring and the staged tree): bulk copies with L2 policies, mbarrier
// waits that suspend in hardware, stage cursors, shared-memory counters.
#pragma once

#include "cluster.cuh"

namespace rra {

// Stage index and mbarrier phase parity of the current message.
struct StagedStage {
  uint32_t b = 0, ph = 0;
  __device__ __forceinline__ void next(int D) {
    if (++b == (uint32_t)D) {
      b = 0;
      ph ^= 1u;
    }
  }
};

// Bulk copy global -> own shared memory with an L2 evict-first policy (the
// input is read once; the FIFO slots should keep their L2 lines).
__device__ __forceinline__ void bulk_load_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], pol;\n\t}" ::"r"(
          cl_smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(cl_smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void red_max_relaxed(uint64_t* p, uint64_t v) {
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_release_cta_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(cl_smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_cta_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(cl_smem_u32(p)) : "memory");
  return v;
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(cl_smem_u32(p)));
  return v;
}

// mbarrier phase wait that suspends the thread in hardware until the phase
// completes or about `hint_ns` pass (so waiting warps take no issue slots);
// false when the time passed first
__device__ __forceinline__ bool mbar_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(cl_smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// mbarrier phase test with CTA-scope acquire (no cluster peers here)
__device__ __forceinline__ bool mbar_try_cta(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(cl_smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbarrier wait bounded by the call's timeout (twice it: a peer wait that
// feeds this one has the same limit) and by the shared abort flag, checked
// each time a suspended wait of up to kStagedSuspendNs gives up.
constexpr uint32_t kStagedSuspendNs = 20000;

__device__ __forceinline__ bool staged_mbar_wait(uint64_t* bar, uint32_t parity, const volatile uint32_t* abort,
                                                 uint64_t timeout_ns) {
  if (mbar_try_cta(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < kMaxSpin; ++it) {
    if (mbar_wait_hint(bar, parity, kStagedSuspendNs)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > 2 * timeout_ns) return false;
  }
  return false;
}

}  // namespace rra
