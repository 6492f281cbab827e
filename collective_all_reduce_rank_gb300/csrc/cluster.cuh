// cluster.cuh -- thread-block-cluster helpers: distributed shared memory
// addresses, cluster barriers, mbarriers with transaction counts, and bulk
// (TMA) copies global <-> shared and shared -> peer shared.
#pragma once

#include "common.cuh"

namespace rra {

__device__ __forceinline__ uint32_t cl_smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of `local` in the CTA of cluster rank `rank`
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(cl_smem_u32(local)), "r"(rank));
  return out;
}

__device__ __forceinline__ void c_mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(cl_smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void c_mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(cl_smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool c_mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(cl_smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait; false when it expired
__device__ __forceinline__ bool c_mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (c_mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0; it < kMaxSpin; ++it) {
    if (c_mbar_try(bar, parity)) return true;
    if ((it & 63u) == 63u && globaltimer() - t0 > timeout_ns) return false;
  }
  return false;
}

__device__ __forceinline__ void c_bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   cl_smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(cl_smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void c_bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(cl_smem_u32(src)),
               "r"(bytes)
               : "memory");
}

// local shared memory -> a peer's shared memory, completing on the peer's
// mbarrier (both peer addresses from mapa)
__device__ __forceinline__ void c_bulk_push(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                            uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(cl_smem_u32(src)), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void c_bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void c_bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void c_bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void c_fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


// remote arrive (release, cluster scope) on a peer's mbarrier
__device__ __forceinline__ void c_mbar_remote_arrive(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

}  // namespace rra
