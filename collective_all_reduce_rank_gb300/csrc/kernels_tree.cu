// kernels_tree.cu -- tree all-reduce on a thread-block cluster.
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Algorithms": tree -- reduce
// up the tree, then broadcast down it, in O(log n) steps; with large
// messages pipelined in chunks its bandwidth is also close to optimal.
//
// One binary tree in heap order over the n virtual ranks (parent of r is
// (r-1)/2, children 2r+1 and 2r+2).  Node r's partial is its own data, then
// its left child's partial, then its right child's:
// p_r = (x_r (+) p_{2r+1}) (+) p_{2r+2}.  Rank 0 rounds the total and it is
// broadcast unchanged, so every rank gets the same bits.
//
// One cluster of n CTAs per channel; cluster CTA r is tree node r.  The
// message is cut into tiles; per batch of G tiles a node
//   up:   waits for its input tile (bulk copy from HBM, prefetched) and its
//         children's partials (pushed into its receive slots), adds them in
//         the order above, and pushes the partial into its parent's slot for
//         this child (the root instead rounds, stores and pushes the result
//         to its children);
//   down: waits for the result from its parent, stores it with a bulk copy
//         and pushes it on to its children.
// Every link is a ring of K slots in the receiver's shared memory; pushes
// are cluster bulk copies completing on the receiver's mbarrier, credits
// come back as remote arrivals on the sender's "slot free" mbarrier.  The
// sub-16-byte tail of the message is summed in the same tree order by one
// thread of the root with plain loads.  Every mbarrier wait is bounded.
#include "cluster.cuh"

namespace rra {

constexpr int kTreeThreads = 256;
constexpr int kTreeXStages = 4;
constexpr int kTreeSlots = 4;

template <int DT>
__host__ __device__ constexpr int tree_tile_units() {
  return Elem<DT>::kAccWords == 2 ? 256 : 512;  // 4 KB of bfloat16, 8 KB of 32-bit data
}

template <int DT>
__host__ __device__ constexpr size_t tree_smem() {
  constexpr size_t T = (size_t)tree_tile_units<DT>() * 16;
  constexpr size_t P = T * Elem<DT>::kAccWords;  // partial tile
  // x stages, up slots from two children, up send slots, down slots, down send slots
  return kTreeXStages * T + 2 * kTreeSlots * P + kTreeSlots * P + kTreeSlots * T + kTreeSlots * T;
}

struct TreeArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  size_t count;  // elements per rank
  int n;
  int channels;
  int G;
  WaitCfg wait;
};

template <int DT>
__device__ void tree_tail(const TreeArgs& a, size_t from) {
  // elements [from, count): fewer than one 16-byte unit, summed in tree order
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.n;
  for (size_t i = from; i < a.count; ++i) {
    float f[kMaxRanks];
    uint32_t u[kMaxRanks];
    for (int r = n - 1; r >= 0; --r) {
      const char* p = static_cast<const char*>(a.in[r]) + i * ES;
      if (DT == RRA_INT32) {
        u[r] = *reinterpret_cast<const uint32_t*>(p);
      } else if (DT == RRA_FLOAT32) {
        f[r] = *reinterpret_cast<const float*>(p);
      } else {
        f[r] = __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(p)) << 16);
      }
      for (int c = 2 * r + 1; c <= 2 * r + 2; ++c) {
        if (c >= n) continue;
        if (DT == RRA_INT32)
          u[r] += u[c];
        else
          f[r] = __fadd_rn(f[r], f[c]);
      }
    }
    for (int r = 0; r < n; ++r) {
      char* q = static_cast<char*>(a.out[r]) + i * ES;
      if (DT == RRA_INT32) {
        *reinterpret_cast<uint32_t*>(q) = u[0];
      } else if (DT == RRA_FLOAT32) {
        *reinterpret_cast<float*>(q) = f[0];
      } else {
        const __nv_bfloat16 h = __float2bfloat16_rn(f[0]);
        *reinterpret_cast<__nv_bfloat16*>(q) = h;
      }
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kTreeThreads, 1) tree_cluster_kernel(const __grid_constant__ TreeArgs a) {
  constexpr int TU = tree_tile_units<DT>();
  constexpr int T = TU * 16;
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int AW = Elem<DT>::kAccWords;
  constexpr int K = kTreeSlots;
  constexpr int XS = kTreeXStages;
  extern __shared__ __align__(128) unsigned char smem[];
  uint4* xbuf = reinterpret_cast<uint4*>(smem);        // [XS][TU]
  uint4* urecv = xbuf + (size_t)XS * TU;               // [2][K][TU*AW]
  uint4* usend = urecv + (size_t)2 * K * TU * AW;      // [K][TU*AW]
  uint4* drecv = usend + (size_t)K * TU * AW;          // [K][TU]
  uint4* dsend = drecv + (size_t)K * TU;               // [K][TU]
  __shared__ __align__(8) uint64_t x_full[XS];
  __shared__ __align__(8) uint64_t u_full[2][K];
  __shared__ __align__(8) uint64_t u_free[K];     // my up-link slots at my parent
  __shared__ __align__(8) uint64_t d_full[K];
  __shared__ __align__(8) uint64_t d_free[2][K];  // my down-link slots at each child
  __shared__ int s_fail;

  const int n = a.n;
  const int r = (int)cluster_rank();
  const int parent = r > 0 ? (r - 1) / 2 : -1;
  const int side = r > 0 ? (r == 2 * parent + 1 ? 0 : 1) : 0;  // which child of the parent
  const bool has_kid[2] = {2 * r + 1 < n, 2 * r + 2 < n};
  const int ch = blockIdx.x / n;
  const int C = a.channels;
  const int G = a.G;
  const int tid = threadIdx.x;
  const size_t units = a.count / PU;
  const size_t per_iter = (size_t)C * G;
  const size_t tiles = (units + TU - 1) / TU;
  const size_t iters = (tiles + per_iter - 1) / per_iter;
  auto tile_of = [&](size_t it, int g) -> size_t { return (it * C + ch) * (size_t)G + g; };
  auto tile_units = [&](size_t t) -> uint32_t {
    const size_t u0 = t * TU;
    return u0 >= units ? 0u : (uint32_t)(units - u0 < (size_t)TU ? units - u0 : (size_t)TU);
  };
  const uint64_t total = (uint64_t)iters * G;  // messages per link (one per tile slot)
  auto msg_tile = [&](uint64_t m) -> size_t { return tile_of((size_t)(m / G), (int)(m % G)); };
  auto issue_x = [&](uint64_t q) {
    if (q >= total) return;
    const uint32_t nu = tile_units(msg_tile(q));
    if (nu == 0) return;
    const int b = (int)(q % XS);
    c_mbar_arrive_tx(&x_full[b], nu * 16u);
    c_bulk_load(xbuf + (size_t)b * TU, static_cast<const char*>(a.in[r]) + msg_tile(q) * (size_t)T, nu * 16u,
                &x_full[b]);
  };

  if (tid == 0) {
    for (int i = 0; i < XS; ++i) c_mbar_init(&x_full[i], 1);
    for (int j = 0; j < K; ++j) {
      c_mbar_init(&u_full[0][j], 2);  // the receiver's arm + the sender's arrival
      c_mbar_init(&u_full[1][j], 2);
      c_mbar_init(&u_free[j], 1);
      c_mbar_init(&d_full[j], 2);
      c_mbar_init(&d_free[0][j], 1);
      c_mbar_init(&d_free[1][j], 1);
    }
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    for (uint64_t m = 0; m < (uint64_t)K && m < total; ++m) {
      const uint32_t nu = tile_units(msg_tile(m));
      for (int s = 0; s < 2; ++s)
        if (has_kid[s]) c_mbar_arrive_tx(&u_full[s][m % K], nu * 16u * AW);
      if (r > 0) c_mbar_arrive_tx(&d_full[m % K], nu * 16u);
    }
    for (int i = 0; i < XS; ++i) issue_x((uint64_t)i);
  }
  cluster_sync();

  const uint64_t tmo = a.wait.timeout_ns;
  auto fail = [&](int idx) {
    if (tid == 0) {
      s_fail = 1;
      record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, idx, 0xFFFFFFFFu);
    }
  };
  uint32_t xphase = 0;
  uint64_t mu = 0, md = 0;  // up / down messages handled
  for (size_t it = 0; it < iters; ++it) {
    // ---- up: reduce this batch's tiles toward the root
    for (int g = 0; g < G; ++g, ++mu) {
      const size_t t = tile_of(it, g);
      const uint32_t nu = tile_units(t);
      const int j = (int)(mu % K);
      const int xb = (int)(mu % XS);
      if (!s_fail && nu > 0) {
        if (!c_mbar_wait(&x_full[xb], (xphase >> xb) & 1u, tmo)) fail((int)mu);
        xphase ^= 1u << xb;
      }
      for (int s = 0; s < 2; ++s)
        if (has_kid[s] && !s_fail && !c_mbar_wait(&u_full[s][j], (uint32_t)(mu / K) & 1u, tmo)) fail((int)mu);
      // the outgoing slot: up to the parent, or (root) down to the children
      if (r > 0) {
        if (mu >= (uint64_t)K && !s_fail && !c_mbar_wait(&u_free[j], (uint32_t)(mu / K - 1) & 1u, tmo)) fail((int)mu);
      } else {
        for (int s = 0; s < 2; ++s)
          if (has_kid[s] && mu >= (uint64_t)K && !s_fail &&
              !c_mbar_wait(&d_free[s][j], (uint32_t)(mu / K - 1) & 1u, tmo))
            fail((int)mu);
      }
      __syncthreads();
      if (!s_fail && nu > 0) {
        const uint4* xs = xbuf + (size_t)xb * TU;
        for (uint32_t u = tid; u < nu; u += kTreeThreads) {
          Acc acc;
          acc_init<DT>(acc, xs[u]);
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            if (!has_kid[s]) continue;
            const uint4* ri = urecv + ((size_t)s * K + j) * TU * AW;
            Acc kid;
            uint4 p[2];
            p[0] = ri[(size_t)u * AW];
            if (AW == 2) p[1] = ri[(size_t)u * AW + 1];
            acc_from_words<DT>(kid, p);
            // acc (+) kid, element by element in the accumulator type
            uint4 w[2];
            acc_to_words<DT>(kid, w);
            if (DT == RRA_INT32) {
              acc.w[0] += w[0].x; acc.w[1] += w[0].y; acc.w[2] += w[0].z; acc.w[3] += w[0].w;
            } else {
#pragma unroll
              for (int e2 = 0; e2 < 4 * AW; ++e2)
                acc.w[e2] = __float_as_uint(__fadd_rn(__uint_as_float(acc.w[e2]), __uint_as_float(kid.w[e2])));
            }
          }
          if (r > 0) {
            uint4 o[2];
            acc_to_words<DT>(acc, o);
            uint4* so = usend + (size_t)j * TU * AW;
            so[(size_t)u * AW] = o[0];
            if (AW == 2) so[(size_t)u * AW + 1] = o[1];
          } else {
            dsend[(size_t)j * TU + u] = acc_narrow<DT>(acc);
          }
        }
        c_fence_proxy_async();
      }
      __syncthreads();
      if (tid == 0 && !s_fail) {
        // every message, empty or not, ends with the sender's arrival on the
        // receiver's barrier: no receiver runs ahead of its sender
        if (r > 0) {
          if (nu > 0)
            c_bulk_push(peer_addr(urecv + ((size_t)side * K + j) * TU * AW, parent), usend + (size_t)j * TU * AW,
                        nu * 16u * AW, peer_addr(&u_full[side][j], parent));
          c_mbar_remote_arrive(peer_addr(&u_full[side][j], parent));
        } else {
          uint4* src = dsend + (size_t)j * TU;
          if (nu > 0) {
            c_bulk_store(static_cast<char*>(a.out[0]) + t * (size_t)T, src, nu * 16u);
            c_bulk_commit();
          }
          for (int s = 0; s < 2; ++s)
            if (has_kid[s]) {
              if (nu > 0)
                c_bulk_push(peer_addr(drecv + (size_t)j * TU, 2 * r + 1 + s), src, nu * 16u,
                            peer_addr(&d_full[j], 2 * r + 1 + s));
              c_mbar_remote_arrive(peer_addr(&d_full[j], 2 * r + 1 + s));
            }
        }
        // children's slots used: re-arm for the message K later, give credits
        for (int s = 0; s < 2; ++s) {
          if (!has_kid[s]) continue;
          if (mu + K < total) c_mbar_arrive_tx(&u_full[s][j], tile_units(msg_tile(mu + K)) * 16u * AW);
          c_mbar_remote_arrive(peer_addr(&u_free[j], 2 * r + 1 + s));
        }
        issue_x(mu + XS);
        if (r == 0 && nu > 0) c_bulk_wait_read0();
      }
    }
    if (r == 0) {
      md += G;  // the root's down messages went out with its up step
      continue;
    }
    // ---- down: the result from the parent, stored and passed on
    for (int g = 0; g < G; ++g, ++md) {
      const size_t t = tile_of(it, g);
      const uint32_t nu = tile_units(t);
      const int j = (int)(md % K);
      if (!s_fail && !c_mbar_wait(&d_full[j], (uint32_t)(md / K) & 1u, tmo)) fail((int)md);
      for (int s = 0; s < 2; ++s)
        if (has_kid[s] && md >= (uint64_t)K && !s_fail &&
            !c_mbar_wait(&d_free[s][j], (uint32_t)(md / K - 1) & 1u, tmo))
          fail((int)md);
      __syncthreads();
      if (!s_fail && nu > 0) {
        const uint4* ri = drecv + (size_t)j * TU;
        uint4* so = dsend + (size_t)j * TU;
        for (uint32_t u = tid; u < nu; u += kTreeThreads) so[u] = ri[u];
        c_fence_proxy_async();
      }
      __syncthreads();
      if (tid == 0 && !s_fail) {
        uint4* src = dsend + (size_t)j * TU;
        if (nu > 0) {
          c_bulk_store(static_cast<char*>(a.out[r]) + t * (size_t)T, src, nu * 16u);
          c_bulk_commit();
        }
        for (int s = 0; s < 2; ++s)
          if (has_kid[s]) {
            if (nu > 0)
              c_bulk_push(peer_addr(drecv + (size_t)j * TU, 2 * r + 1 + s), src, nu * 16u,
                          peer_addr(&d_full[j], 2 * r + 1 + s));
            c_mbar_remote_arrive(peer_addr(&d_full[j], 2 * r + 1 + s));
          }
        if (md + K < total) c_mbar_arrive_tx(&d_full[j], tile_units(msg_tile(md + K)) * 16u);
        c_mbar_remote_arrive(peer_addr(&d_free[side][j], parent));
        if (nu > 0) c_bulk_wait_read0();
      }
    }
  }
  if (tid == 0) {
    c_bulk_wait0();
    if (r == 0 && ch == 0 && !s_fail) tree_tail<DT>(a, units * PU);
  }
  __syncthreads();
  cluster_sync();
}

template <int DT>
static cudaError_t tree_go(const TreeArgs& a, int grid, cudaStream_t s) {
  constexpr size_t smem = tree_smem<DT>();
  static const cudaError_t attr =
      cudaFuncSetAttribute(tree_cluster_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = a.n;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_cluster_kernel<DT>, a);
}

template <int DT>
static int tree_clusters(int n) {
  constexpr size_t smem = tree_smem<DT>();
  cudaFuncSetAttribute(tree_cluster_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n * 64);
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = n;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, tree_cluster_kernel<DT>, &cfg) != cudaSuccess) return 0;
  return clusters;
}

int tree_tile_units_for(int dt) { return dt == RRA_BFLOAT16 ? tree_tile_units<RRA_BFLOAT16>() : tree_tile_units<RRA_FLOAT32>(); }

int tree_max_clusters(int n, int dt) {
  if (n < 2 || n > kMaxRanks) return 0;
  if (dt == RRA_INT32) return tree_clusters<RRA_INT32>(n);
  if (dt == RRA_FLOAT32) return tree_clusters<RRA_FLOAT32>(n);
  return tree_clusters<RRA_BFLOAT16>(n);
}

cudaError_t launch_tree(int dt, const void* const* in, void* const* out, int n, size_t count, int channels, int G,
                        const WaitCfg& w, cudaStream_t s) {
  TreeArgs a{};
  for (int r = 0; r < n; ++r) {
    a.in[r] = in[r];
    a.out[r] = out[r];
  }
  a.count = count;
  a.n = n;
  a.channels = channels;
  a.G = G;
  a.wait = w;
  if (dt == RRA_INT32) return tree_go<RRA_INT32>(a, n * channels, s);
  if (dt == RRA_FLOAT32) return tree_go<RRA_FLOAT32>(a, n * channels, s);
  return tree_go<RRA_BFLOAT16>(a, n * channels, s);
}

}  // namespace rra
