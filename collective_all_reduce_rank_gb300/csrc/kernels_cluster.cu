// kernels_cluster.cu -- two-shot all-reduce on a thread-block cluster.
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Algorithms": two-shot --
// each rank reads its 1/n of the other ranks' data and sums it (a
// reduce-scatter), then reads the sums back (an all-gather); two
// synchronizations.
//
// One cluster of n CTAs per channel: cluster CTA r is virtual rank r.  Per
// iteration, for tile t of every chunk:
//   1. the n input tiles of chunk r stream from HBM into shared memory by
//      bulk copies (two stages, prefetched two iterations ahead);
//   2. the CTA sums them (ascending rank order) into its reduced tile and
//      writes it to outs[r] with a bulk store;
//   3. it pushes the reduced tile into every peer's shared memory with a
//      cluster bulk copy that completes on the peer's mbarrier (the
//      all-gather read of the reduced slice, through distributed shared
//      memory instead of HBM);
//   4. once the n-1 peer tiles have arrived on its own mbarrier, it writes
//      them to outs[r] with bulk stores.
// The two synchronizations of two-shot are the cluster barrier at the top
// of each iteration (every peer's gather buffer is free and its barrier
// armed) and the mbarrier the pushes complete on.  HBM sees each input once
// and each output once.  Whole 16-byte units only: the host finishes a
// ragged tail (fewer than 16 bytes) with the one-shot kernel, same bits.
//
// Bounded waits: every mbarrier wait gives up after the call's timeout,
// records RRA_ERR_TIMEOUT and skips the work, but the CTA keeps taking the
// cluster barriers so its peers never wait on it forever.
#include "cluster.cuh"

namespace rra {

constexpr int kClusterThreads = 256;

template <int N>
__host__ __device__ constexpr int c2_tile() {
  return N <= 4 ? 16384 : 8192;
}
template <int N>
__host__ __device__ constexpr size_t c2_smem() {
  return (size_t)(2 * N + 1 + N) * c2_tile<N>();  // in[2][N] + red + gat[N]
}

template <int N, int DT>
__global__ void __launch_bounds__(kClusterThreads, 1)
    twoshot_cluster_kernel(const __grid_constant__ TwoShotArgs a) {
  constexpr int T = c2_tile<N>();
  constexpr int TU = T / 16;
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int ES = Elem<DT>::kSize;
  extern __shared__ __align__(128) unsigned char smem[];
  uint4* in = reinterpret_cast<uint4*>(smem);                     // [2][N][TU]
  uint4* red = in + (size_t)2 * N * TU;                           // [TU]
  uint4* gat = red + TU;                                          // [N][TU] (own slot unused)
  __shared__ __align__(8) uint64_t full_in[2];
  __shared__ __align__(8) uint64_t full_gat;
  __shared__ int s_fail;

  const int r = (int)cluster_rank();
  const int ch = blockIdx.x / N;
  const int C = a.channels;
  const int tid = threadIdx.x;
  // whole units per chunk (a ragged tail is not part of this kernel)
  auto units = [&](int c) -> size_t { return a.chunk_len[c] / PU; };
  auto tile_units = [&](int c, size_t i) -> uint32_t {
    const size_t u0 = (i * C + ch) * (size_t)TU;
    const size_t uc = units(c);
    return u0 >= uc ? 0u : (uint32_t)(uc - u0 < (size_t)TU ? uc - u0 : (size_t)TU);
  };
  auto chunk_ptr = [&](const void* base, int c, size_t i) -> const char* {
    return static_cast<const char*>(base) + a.chunk_lo[c] * ES + (i * C + ch) * (size_t)T;
  };
  const size_t iters = (units(0) + (size_t)C * TU - 1) / ((size_t)C * TU);

  if (tid == 0) {
    c_mbar_init(&full_in[0], 1);
    c_mbar_init(&full_in[1], 1);
    c_mbar_init(&full_gat, 1);
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_sync();  // every peer's barriers exist before anyone pushes

  auto issue_inputs = [&](size_t i) {
    const uint32_t nu = tile_units(r, i);
    if (nu == 0) return;
    const int s = (int)(i & 1);
    c_mbar_arrive_tx(&full_in[s], nu * 16u * N);
#pragma unroll
    for (int k = 0; k < N; ++k) c_bulk_load(in + ((size_t)s * N + k) * TU, chunk_ptr(a.in[k], r, i), nu * 16u, &full_in[s]);
  };
  if (tid == 0) {
    issue_inputs(0);
    if (iters > 1) issue_inputs(1);
  }

  for (size_t i = 0; i < iters; ++i) {
    const int s = (int)(i & 1);
    const uint32_t nu = tile_units(r, i);
    // arm the gather barrier with the bytes the peers will push this time
    if (tid == 0) {
      c_bulk_wait_read0();  // last iteration's stores have read red and gat
      uint32_t bytes = 0;
#pragma unroll
      for (int q = 0; q < N; ++q)
        if (q != r) bytes += tile_units(q, i) * 16u;
      c_mbar_arrive_tx(&full_gat, bytes);
    }
    cluster_sync();  // sync 1: peers armed, gather buffers free

    // reduce-scatter part: sum the n input tiles of chunk r
    if (nu > 0) {
      bool ok = c_mbar_wait(&full_in[s], (uint32_t)(i >> 1) & 1u, a.wait.timeout_ns);
      if (!ok && tid == 0) {
        s_fail = 1;
        record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, (int)i, 0xFFFFFFFFu);
      }
      const uint4* st = in + (size_t)s * N * TU;
      if (ok) {
        for (uint32_t u = tid; u < nu; u += kClusterThreads) {
          Acc acc;
          acc_init<DT>(acc, st[u]);
#pragma unroll
          for (int k = 1; k < N; ++k) acc_add<DT>(acc, st[(size_t)k * TU + u]);
          red[u] = acc_narrow<DT>(acc);
        }
      }
      c_fence_proxy_async();
    }
    __syncthreads();
    if (tid == 0) {
      if (nu > 0) {
        c_bulk_store(const_cast<char*>(chunk_ptr(a.out[r], r, i)), red, nu * 16u);
        c_bulk_commit();
        // all-gather part: push the reduced tile into every peer's slot r
#pragma unroll
        for (int q = 0; q < N; ++q)
          if (q != r)
            c_bulk_push(peer_addr(gat + (size_t)r * TU, q), red, nu * 16u, peer_addr(&full_gat, q));
      }
      if (i + 2 < iters) issue_inputs(i + 2);  // stage s is free: everyone is past the sum
      // sync 2: the peers' tiles have arrived
      if (!c_mbar_wait(&full_gat, (uint32_t)i & 1u, a.wait.timeout_ns)) {
        s_fail = 1;
        record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, (int)i, 0xFFFFFFFFu);
      } else {
#pragma unroll
        for (int q = 0; q < N; ++q) {
          const uint32_t nq = tile_units(q, i);
          if (q != r && nq > 0) c_bulk_store(const_cast<char*>(chunk_ptr(a.out[r], q, i)), gat + (size_t)q * TU, nq * 16u);
        }
        c_bulk_commit();
      }
    }
    __syncthreads();
  }
  if (tid == 0) c_bulk_wait0();
  __syncthreads();
  cluster_sync();  // no CTA leaves while a peer may still push into it
}

template <int N, int DT>
static cudaError_t c2_go(const TwoShotArgs& a, int grid, cudaStream_t s) {
  constexpr size_t smem = c2_smem<N>();
  static const cudaError_t attr = cudaFuncSetAttribute(twoshot_cluster_kernel<N, DT>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = N;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, twoshot_cluster_kernel<N, DT>, a);
}

template <int N, int DT>
static int c2_max_clusters() {
  constexpr size_t smem = c2_smem<N>();
  cudaFuncSetAttribute(twoshot_cluster_kernel<N, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(N * 64);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = N;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, twoshot_cluster_kernel<N, DT>, &cfg) != cudaSuccess) return 0;
  return clusters;
}

template <int N>
static cudaError_t c2_n(int dt, const TwoShotArgs& a, int grid, cudaStream_t s) {
  if (dt == RRA_INT32) return c2_go<N, RRA_INT32>(a, grid, s);
  if (dt == RRA_FLOAT32) return c2_go<N, RRA_FLOAT32>(a, grid, s);
  return c2_go<N, RRA_BFLOAT16>(a, grid, s);
}

template <int N>
static int c2_clusters_n(int dt) {
  if (dt == RRA_INT32) return c2_max_clusters<N, RRA_INT32>();
  if (dt == RRA_FLOAT32) return c2_max_clusters<N, RRA_FLOAT32>();
  return c2_max_clusters<N, RRA_BFLOAT16>();
}

int twoshot_cluster_tile_bytes(int n) { return n <= 4 ? c2_tile<4>() : c2_tile<8>(); }

int twoshot_cluster_max_clusters(int n, int dt) {
  switch (n) {
    case 2: return c2_clusters_n<2>(dt);
    case 3: return c2_clusters_n<3>(dt);
    case 4: return c2_clusters_n<4>(dt);
    case 5: return c2_clusters_n<5>(dt);
    case 6: return c2_clusters_n<6>(dt);
    case 7: return c2_clusters_n<7>(dt);
    case 8: return c2_clusters_n<8>(dt);
    default: return 0;
  }
}

cudaError_t launch_twoshot_cluster(int n, int dt, const TwoShotArgs& a, int grid, cudaStream_t s) {
  switch (n) {
    case 2: return c2_n<2>(dt, a, grid, s);
    case 3: return c2_n<3>(dt, a, grid, s);
    case 4: return c2_n<4>(dt, a, grid, s);
    case 5: return c2_n<5>(dt, a, grid, s);
    case 6: return c2_n<6>(dt, a, grid, s);
    case 7: return c2_n<7>(dt, a, grid, s);
    case 8: return c2_n<8>(dt, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rra
