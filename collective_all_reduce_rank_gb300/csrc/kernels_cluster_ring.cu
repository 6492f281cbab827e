// kernels_cluster_ring.cu -- the ring on a thread-block cluster.
//
// Same schedule and summation order as kernels_ring.cu ("NCCL collectives,
// ring all-reduce & launching TP/PP", "Direct answer" and "Deep dive";
// "Collective communication: NCCL's algorithms and protocols...",
// "Algorithms"): n-1 reduce-scatter steps, in which rank r sends the partial
// of chunk (r-s-1) to r+1 which adds its own slice, then n-1 all-gather
// steps forwarding the reduced chunks; chunk c is summed x_{c+1}, ..., x_c.
//
// One cluster of n CTAs per channel; cluster CTA r is virtual rank r and
// the link r -> r+1 is a ring of K receive slots in CTA r+1's shared
// memory:
//   - CTA r builds each outgoing message (a tile of T input bytes: a
//     float32-accumulator partial during the reduce-scatter, final values
//     during the all-gather) in a local send slot and pushes it into slot
//     m mod K of CTA r+1 with a cluster bulk copy that completes on CTA
//     r+1's mbarrier for that slot;
//   - CTA r+1, once it has used the slot, re-arms that mbarrier for the
//     message K later and arrives remotely on CTA r's "slot free" mbarrier,
//     which CTA r waits on before it pushes into the slot again (credits).
// The rank's own input tiles stream from HBM into shared memory with bulk
// copies, several messages ahead; final values go to HBM with bulk stores.
// Each step moves G tiles, so the message a rank needs next was pushed G
// messages earlier.  HBM sees each input once and each output once; the
// links never touch it.  Whole 16-byte units only (the host finishes a
// ragged tail with a rotated one-shot sum, same order and bits).
//
// Every mbarrier wait is bounded; on expiry the CTA records RRA_ERR_TIMEOUT
// and stops working, but still takes the final cluster barrier.
#include "cluster.cuh"

namespace rra {

constexpr int kCRingThreads = 256;
constexpr int kCRingXStages = 4;

struct CRingShape {
  int K;  // receive / send slots per link
  int G;  // tiles per step
};

template <int DT>
__host__ __device__ constexpr int cring_tile() {  // input bytes per message
  return 8192;
}

template <int DT>
__host__ __device__ constexpr int cring_slots() {
  return Elem<DT>::kAccWords == 2 ? 4 : 8;
}

template <int DT>
__host__ __device__ constexpr size_t cring_smem() {
  // x stages + K receive slots + K send slots (slots sized for accumulators)
  // + one output tile for steps that store without sending
  return (size_t)kCRingXStages * cring_tile<DT>() +
         (size_t)2 * cring_slots<DT>() * cring_tile<DT>() * Elem<DT>::kAccWords + cring_tile<DT>();
}

template <int DT>
__global__ void __launch_bounds__(kCRingThreads, 1) ring_cluster_kernel(const __grid_constant__ RingArgs a) {
  constexpr int T = cring_tile<DT>();
  constexpr int TU = T / 16;
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int ES = Elem<DT>::kSize;
  constexpr int AW = Elem<DT>::kAccWords;
  constexpr int K = cring_slots<DT>();
  constexpr int XS = kCRingXStages;
  const int G = a.G;
  extern __shared__ __align__(128) unsigned char smem[];
  uint4* xbuf = reinterpret_cast<uint4*>(smem);  // [XS][TU]
  uint4* rslot = xbuf + (size_t)XS * TU;         // [K][TU * AW]
  uint4* sslot = rslot + (size_t)K * TU * AW;    // [K][TU * AW]
  uint4* obuf = sslot + (size_t)K * TU * AW;     // [TU]: output of a step that does not send
  __shared__ __align__(8) uint64_t x_full[XS];
  __shared__ __align__(8) uint64_t r_full[K];
  __shared__ __align__(8) uint64_t s_free[K];
  __shared__ int s_fail;

  const int n = a.n;
  const int r = (int)cluster_rank();
  const int prev = (r + n - 1) % n, next = (r + 1) % n;
  const int ch = blockIdx.x / n;
  const int C = a.channels;
  const int tid = threadIdx.x;
  const int mode = a.mode;
  // sends (= receives) per iteration and the chunk each send carries
  const int S = mode == kRingAllReduce ? 2 * (n - 1) : n - 1;
  auto send_chunk = [&](int rank, int k) -> int {
    if (mode == kRingAllGather) return ((rank - k) % n + n) % n;
    if (k <= n - 2) return ((rank - k - 1) % n + n) % n;
    if (k == n - 1) return rank;
    return ((rank - (k - n + 1)) % n + n) % n;
  };
  auto tile_units = [&](int c, size_t tile) -> uint32_t {
    const size_t uc = a.len[c] / PU;
    const size_t u0 = tile * TU;
    return u0 >= uc ? 0u : (uint32_t)(uc - u0 < (size_t)TU ? uc - u0 : (size_t)TU);
  };
  size_t maxu = 0;
  for (int c = 0; c < n; ++c) maxu = a.len[c] / PU > maxu ? a.len[c] / PU : maxu;
  const size_t tiles_per_iter = (size_t)C * G;
  const size_t iters = (maxu + tiles_per_iter * TU - 1) / (tiles_per_iter * TU);
  auto tile_of = [&](size_t it, int g) -> size_t { return (it * C + ch) * (size_t)G + g; };
  const uint64_t total_msgs = (uint64_t)iters * S * G;
  // message m (in or out) -> iteration, step, tile
  auto msg_units = [&](int rank, uint64_t m) -> uint32_t {
    const size_t it = (size_t)(m / ((uint64_t)S * G));
    const int rem = (int)(m % ((uint64_t)S * G));
    return tile_units(send_chunk(rank, rem / G), tile_of(it, rem % G));
  };
  // x tiles this rank reads, in order: RS sends 0..n-2 and the final step
  // (chunk r), or in all-gather mode only the own shard
  const int XP = mode == kRingAllGather ? 1 : n;  // x reads per tile position
  auto x_chunk = [&](int p) -> int { return mode == kRingAllGather ? r : (p <= n - 2 ? ((r - p - 1) % n + n) % n : r); };
  const uint64_t total_x = (uint64_t)iters * XP * G;
  auto x_units = [&](uint64_t q) -> uint32_t {
    const size_t it = (size_t)(q / ((uint64_t)XP * G));
    const int rem = (int)(q % ((uint64_t)XP * G));
    return tile_units(x_chunk(rem / G), tile_of(it, rem % G));
  };
  auto x_ptr = [&](uint64_t q) -> const char* {
    const size_t it = (size_t)(q / ((uint64_t)XP * G));
    const int rem = (int)(q % ((uint64_t)XP * G));
    const int c = x_chunk(rem / G);
    return static_cast<const char*>(a.in[r]) + a.ibase[c] * ES + tile_of(it, rem % G) * (size_t)T;
  };
  auto issue_x = [&](uint64_t q) {
    if (q >= total_x) return;
    const uint32_t nu = x_units(q);
    if (nu == 0) return;
    const int b = (int)(q % XS);
    c_mbar_arrive_tx(&x_full[b], nu * 16u);
    c_bulk_load(xbuf + (size_t)b * TU, x_ptr(q), nu * 16u, &x_full[b]);
  };
  auto arm_recv = [&](uint64_t m) {
    if (m >= total_msgs) return;
    const uint32_t nu = msg_units(prev, m);
    const int rem = (int)(m % ((uint64_t)S * G)) / G;  // prev's send index: partial or final words
    const bool partial = mode != kRingAllGather && rem <= n - 2;
    c_mbar_arrive_tx(&r_full[m % K], nu * 16u * (partial ? AW : 1));
  };

  if (tid == 0) {
    for (int i = 0; i < XS; ++i) c_mbar_init(&x_full[i], 1);
    for (int j = 0; j < K; ++j) {
      c_mbar_init(&r_full[j], 2);  // the receiver's arm + the sender's arrival
      c_mbar_init(&s_free[j], 1);
    }
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    for (int j = 0; j < K; ++j) arm_recv((uint64_t)j);
    for (int i = 0; i < XS; ++i) issue_x((uint64_t)i);
  }
  cluster_sync();  // every CTA's barriers armed before any push

  uint64_t m_in = 0, m_out = 0, xq = 0;
  uint32_t xphase = 0;  // bit b: parity of x buffer b's next wait
  const uint64_t tmo = a.wait.timeout_ns;
  auto fail = [&](int idx) {
    if (tid == 0) {
      s_fail = 1;
      record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, idx, 0xFFFFFFFFu);
    }
  };

  for (size_t it = 0; it < iters; ++it) {
    // actions of this iteration: index k over sends+receives in schedule order
    // AR: k=0 send-only, 1..n-2 recv+send (RS), n-1 recv+final+send,
    //     n..2n-3 recv+store+send (AG), 2n-2 recv+store (last)
    // RS: 0 send, 1..n-2 recv+send, n-1 recv+final
    // AG: 0 own shard store+send, 1..n-2 recv+store+send, n-1 recv+store
    const int actions = mode == kRingAllReduce ? 2 * n - 1 : n;
    for (int k = 0; k < actions; ++k) {
      const bool recv = k > 0;
      const bool send = mode == kRingAllReduce ? k < 2 * n - 2 : k < n - 1;
      const bool uses_x = mode == kRingAllGather ? k == 0 : k <= n - 1;
      const bool final_rs = mode != kRingAllGather && k == n - 1;
      const bool ag_store = mode == kRingAllGather ? true : (mode == kRingAllReduce && k >= n);
      const bool partial_out = send && mode != kRingAllGather && k <= n - 2;
      // chunk this action stores / reduces
      const int c = mode == kRingAllGather ? ((r - k) % n + n) % n
                                           : (k <= n - 2 ? ((r - k - 1) % n + n) % n
                                                         : (k == n - 1 ? r : ((r - (k - n + 1)) % n + n) % n));
      for (int g = 0; g < G; ++g) {
        const size_t tile = tile_of(it, g);
        const uint32_t nu = tile_units(c, tile);
        int xb = -1;
        if (uses_x) {
          if (nu > 0 && !s_fail) {
            xb = (int)(xq % XS);
            if (!c_mbar_wait(&x_full[xb], (xphase >> xb) & 1u, tmo)) fail((int)xq);
            xphase ^= 1u << xb;
          }
        }
        const int jin = (int)(m_in % K), jout = (int)(m_out % K);
        if (recv && !s_fail && !c_mbar_wait(&r_full[jin], (uint32_t)(m_in / K) & 1u, tmo)) fail((int)m_in);
        if (send && m_out >= (uint64_t)K && !s_fail &&
            !c_mbar_wait(&s_free[jout], (uint32_t)(m_out / K - 1) & 1u, tmo))
          fail((int)m_out);
        __syncthreads();
        // a step that sends builds its message in the send slot (free: its
        // credit came back); one that only stores uses the output tile
        uint4* so = send ? sslot + (size_t)jout * TU * AW : obuf;
        if (!s_fail && nu > 0) {
          const uint4* xs = xb >= 0 ? xbuf + (size_t)xb * TU : nullptr;
          const uint4* ri = rslot + (size_t)jin * TU * AW;
          for (uint32_t u = tid; u < nu; u += kCRingThreads) {
            if (partial_out || final_rs) {
              Acc acc;
              if (!recv) {
                acc_init<DT>(acc, xs[u]);
              } else {
                uint4 p[2];
                p[0] = ri[(size_t)u * AW];
                if (AW == 2) p[1] = ri[(size_t)u * AW + 1];
                acc_from_words<DT>(acc, p);
                acc_add<DT>(acc, xs[u]);
              }
              if (final_rs) {
                so[u] = acc_narrow<DT>(acc);  // final values: one word per unit
              } else {
                uint4 o[2];
                acc_to_words<DT>(acc, o);
                so[(size_t)u * AW] = o[0];
                if (AW == 2) so[(size_t)u * AW + 1] = o[1];
              }
            } else if (mode == kRingAllGather && k == 0) {
              so[u] = xs[u];
            } else {
              so[u] = ri[u];  // all-gather: forward / store the final values
            }
          }
          c_fence_proxy_async();
        }
        __syncthreads();
        if (tid == 0 && !s_fail) {
          if (nu > 0 && (final_rs || ag_store)) {
            char* y = static_cast<char*>(a.out[r]) + a.obase[c] * ES + tile * (size_t)T;
            c_bulk_store(y, so, nu * 16u);
            c_bulk_commit();
          }
          if (send) {
            if (nu > 0) {
              const uint32_t bytes = nu * 16u * (partial_out ? AW : 1);
              c_bulk_push(peer_addr(rslot + (size_t)jout * TU * AW, next), so, bytes, peer_addr(&r_full[jout], next));
            }
            // the sender's arrival, also for an empty tile: the receiver never
            // consumes (and credits) a message its sender has not reached
            c_mbar_remote_arrive(peer_addr(&r_full[jout], next));
          }
          if (recv) {
            arm_recv(m_in + K);  // before the credit: the next push into this slot finds it armed
            c_mbar_remote_arrive(peer_addr(&s_free[jin], prev));
          }
          // x tile xq is used (or was empty): its buffer takes tile xq + XS
          if (uses_x) issue_x(xq + XS);
          if (nu > 0 && (final_rs || ag_store)) c_bulk_wait_read0();  // slot / tile reusable
        }
        if (uses_x) ++xq;
        if (recv) ++m_in;
        if (send) ++m_out;
      }
    }
  }
  if (tid == 0) c_bulk_wait0();
  __syncthreads();
  cluster_sync();  // pushes into and credits to every CTA have landed
}

template <int DT>
static cudaError_t cring_go(const RingArgs& a, int grid, cudaStream_t s) {
  constexpr size_t smem = cring_smem<DT>();
  static const cudaError_t attr =
      cudaFuncSetAttribute(ring_cluster_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCRingThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = a.n;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ring_cluster_kernel<DT>, a);
}

template <int DT>
static int cring_clusters(int n) {
  constexpr size_t smem = cring_smem<DT>();
  cudaFuncSetAttribute(ring_cluster_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n * 64);
  cfg.blockDim = dim3(kCRingThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = n;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, ring_cluster_kernel<DT>, &cfg) != cudaSuccess) return 0;
  return clusters;
}

int ring_cluster_tile_units(int dt) { return dt == RRA_BFLOAT16 ? cring_tile<RRA_BFLOAT16>() / 16 : cring_tile<RRA_FLOAT32>() / 16; }
int ring_cluster_slots(int dt) { return dt == RRA_BFLOAT16 ? cring_slots<RRA_BFLOAT16>() : cring_slots<RRA_FLOAT32>(); }

int ring_cluster_max_clusters(int n, int dt) {
  if (n < 2 || n > kMaxRanks) return 0;
  if (dt == RRA_INT32) return cring_clusters<RRA_INT32>(n);
  if (dt == RRA_FLOAT32) return cring_clusters<RRA_FLOAT32>(n);
  return cring_clusters<RRA_BFLOAT16>(n);
}

cudaError_t launch_ring_cluster(int dt, const RingArgs& a, int grid, cudaStream_t s) {
  if (dt == RRA_INT32) return cring_go<RRA_INT32>(a, grid, s);
  if (dt == RRA_FLOAT32) return cring_go<RRA_FLOAT32>(a, grid, s);
  return cring_go<RRA_BFLOAT16>(a, grid, s);
}

}  // namespace rra
