// kernels_tma.cu -- one-shot all-reduce with bulk-copy (TMA) staging.
//
// Same result and summation order as oneshot_kernel (ascending rank order,
// every rank's output the same bits), different data movement: a persistent
// CTA per SM streams tiles of the n inputs into a ring of shared-memory
// stages with cp.async.bulk (completion counted on an mbarrier), its threads
// sum the n tiles out of shared memory into an output tile, and one thread
// writes that tile to all n outputs with n bulk stores.  The copy engine of
// the SM (not the LSU) moves every byte; the threads only add.
//
// Every mbarrier wait is bounded (iteration cap and %globaltimer); on
// expiry the CTA records RRA_ERR_TIMEOUT (when a status block is given),
// waits for its own bulk stores to finish reading shared memory, and
// returns.
#include <algorithm>

#include "common.cuh"

namespace rra {

constexpr int kTmaThreads = 256;
constexpr int kTmaTile = 8192;  // bytes per input per stage
constexpr int kTmaSmemBudget = 200 * 1024;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct TmaArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  size_t units;       // whole 16-byte units handled here (the tail is elsewhere)
  DevStatus* status;  // may be null
  uint64_t timeout_ns;
};

template <int N>
__host__ __device__ constexpr int tma_stages() {
  return (kTmaSmemBudget - 2 * kTmaTile) / (N * kTmaTile) < 8 ? (kTmaSmemBudget - 2 * kTmaTile) / (N * kTmaTile)
                                                                : 8;
}

template <int N, int DT>
__global__ void __launch_bounds__(kTmaThreads, 1) oneshot_tma_kernel(const __grid_constant__ TmaArgs a) {
  constexpr int S = tma_stages<N>();
  constexpr int TU = kTmaTile / 16;  // units per tile
  extern __shared__ __align__(128) unsigned char smem[];
  uint4* stage = reinterpret_cast<uint4*>(smem);                        // [S][N][TU]
  uint4* obuf = reinterpret_cast<uint4*>(smem + (size_t)S * N * kTmaTile);  // [2][TU]
  __shared__ __align__(8) uint64_t full[S];
  __shared__ int s_fail;

  const size_t tiles = (a.units + TU - 1) / TU;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  auto tile_units = [&](size_t t) -> uint32_t {
    const size_t left = a.units - t * TU;
    return (uint32_t)(left < (size_t)TU ? left : (size_t)TU);
  };
  auto issue = [&](size_t t, int s) {
    const uint32_t bytes = tile_units(t) * 16u;
    mbar_expect_tx(&full[s], bytes * N);
#pragma unroll
    for (int k = 0; k < N; ++k)
      bulk_load(stage + ((size_t)s * N + k) * TU, static_cast<const char*>(a.in[k]) + t * (size_t)kTmaTile,
                bytes, &full[s]);
  };

  // prologue: fill the stages
  size_t t = blockIdx.x;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      const size_t tt = t + (size_t)s * gridDim.x;
      if (tt < tiles) issue(tt, s);
    }
  }
  uint32_t i = 0;
  for (; t < tiles; t += gridDim.x, ++i) {
    const int s = (int)(i % S);
    const uint32_t parity = (i / S) & 1u;
    // bounded wait for the stage's bytes
    if (tid == 0) {
      bool ok = false;
      const uint64_t t0 = globaltimer();
      for (uint32_t it = 0; it < kMaxSpin; ++it) {
        if (mbar_try_wait(&full[s], parity)) { ok = true; break; }
        if ((it & 63u) == 63u && globaltimer() - t0 > a.timeout_ns) break;
      }
      if (!ok) {
        s_fail = 1;
        if (a.status) record_error(a.status, RRA_ERR_TIMEOUT, blockIdx.x, -1, (int)t, 0xFFFFFFFFu);
      }
    }
    __syncthreads();
    if (s_fail) break;
    // every thread observes the completed phase too (it has completed:
    // thread 0 saw it, and only thread 0 re-arms it, later), which orders
    // the bulk-copy writes before this thread's reads
    for (uint32_t it = 0; it < kMaxSpin && !mbar_try_wait(&full[s], parity); ++it) {
    }
    const int ob = (int)(i & 1u);
    if (i >= 2) {
      // the stores of tile i-2 read obuf[ob]; at most one group (tile i-1)
      // may still be reading
      if (tid == 0) bulk_wait_read<1>();
      __syncthreads();
    }
    const uint32_t nu = tile_units(t);
    const uint4* st = stage + (size_t)s * N * TU;
    uint4* o = obuf + (size_t)ob * TU;
    for (uint32_t u = tid; u < nu; u += kTmaThreads) {
      Acc acc;
      acc_init<DT>(acc, st[u]);
#pragma unroll
      for (int k = 1; k < N; ++k) acc_add<DT>(acc, st[(size_t)k * TU + u]);
      o[u] = acc_narrow<DT>(acc);
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int r = 0; r < N; ++r) bulk_store(static_cast<char*>(a.out[r]) + t * (size_t)kTmaTile, o, nu * 16u);
      bulk_commit();
      const size_t nt = t + (size_t)S * gridDim.x;
      if (nt < tiles) issue(nt, s);  // the stage was fully read before the barrier above
    }
  }
  if (tid == 0) bulk_wait_all();
  __syncthreads();
}

template <int N, int DT>
static cudaError_t tma_go(const TmaArgs& a, int* grid, cudaStream_t s) {
  constexpr int S = tma_stages<N>();
  const size_t smem = (size_t)S * N * kTmaTile + 2 * kTmaTile;
  static const cudaError_t attr =
      cudaFuncSetAttribute(oneshot_tma_kernel<N, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return attr;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t tiles = (a.units + kTmaTile / 16 - 1) / (kTmaTile / 16);
  *grid = (int)std::max<size_t>(1, std::min<size_t>(tiles, (size_t)sms));
  oneshot_tma_kernel<N, DT><<<*grid, kTmaThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int N>
static cudaError_t tma_n(int dt, const TmaArgs& a, int* grid, cudaStream_t s) {
  if (dt == RRA_INT32) return tma_go<N, RRA_INT32>(a, grid, s);
  if (dt == RRA_FLOAT32) return tma_go<N, RRA_FLOAT32>(a, grid, s);
  return tma_go<N, RRA_BFLOAT16>(a, grid, s);
}

cudaError_t launch_oneshot_tma(int n, int dt, const void* const* in, void* const* out, size_t units,
                               DevStatus* status, uint64_t timeout_ns, int* grid, cudaStream_t s) {
  TmaArgs a{};
  for (int r = 0; r < n; ++r) {
    a.in[r] = in[r];
    a.out[r] = out[r];
  }
  a.units = units;
  a.status = status;
  a.timeout_ns = timeout_ns;
  switch (n) {
    case 1: return tma_n<1>(dt, a, grid, s);
    case 2: return tma_n<2>(dt, a, grid, s);
    case 3: return tma_n<3>(dt, a, grid, s);
    case 4: return tma_n<4>(dt, a, grid, s);
    case 5: return tma_n<5>(dt, a, grid, s);
    case 6: return tma_n<6>(dt, a, grid, s);
    case 7: return tma_n<7>(dt, a, grid, s);
    case 8: return tma_n<8>(dt, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rra
