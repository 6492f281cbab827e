// kernels_ring.cu -- ring all-reduce and its reduce-scatter / all-gather
// halves.
//
// "NCCL collectives, ring all-reduce & launching TP/PP", sections "Direct
// answer" and "Deep dive": ring all-reduce = reduce-scatter + all-gather;
// the ring pipelines the data in N chunks so every link is busy.
// "Collective communication: NCCL's algorithms and protocols...", section
// "Algorithms": n-1 reduce-scatter steps and n-1 all-gather steps, each
// GPU sending and receiving 2(n-1)/n S.
//
// Schedule, per rank r (indices mod n):
//   RS step s = 0..n-2: send the partial of chunk (r-s-1) to r+1; the
//     receiver adds its own slice of that chunk.  Rank r ends with chunk r,
//     summed x_{r+1}, x_{r+2}, ..., x_{r-1}, x_r.
//   AG step s = 0..n-2: forward chunk (r-s) to r+1, which stores it.
//
// Design on one GPU: one persistent cooperative launch of n x C CTAs; CTA
// (r, ch) is channel ch of virtual rank r and every one of its 16 warps is
// an independent pipeline.  The link r -> r+1 of (channel, warp) is a
// FIFO of K slots in the workspace, small enough to stay in L2, with a head
// counter (messages posted by the sender) and a tail counter (messages
// consumed by the receiver).  Send = write the slot, __syncwarp, release
// the head (data -> fence -> flag: the Simple protocol of the page's
// "Protocols" section); receive = acquire the head, read the slot, release
// the tail.  Each step moves G slices of the channel's part of a chunk;
// the receiver of slice g in step s+1 needs slice g of step s, posted G
// messages earlier, so the flag latency hides behind the other slices.
// bfloat16 partial sums travel as float32 and are rounded once, at the
// final reduce-scatter step.  Only the inputs are read from HBM and only
// the outputs written to it; the slots stay in L2.
#include "common.cuh"

namespace rra {

template <int DT, bool VEC>
struct RingWarp {
  static constexpr int PU = Elem<DT>::kPerUnit;
  static constexpr int ES = Elem<DT>::kSize;
  static constexpr int AW = Elem<DT>::kAccWords;
  static constexpr int UPT = kRingUnitsPerThread;

  const RingArgs& a;
  int r, prev, next, lane;
  uint64_t E;
  uint32_t tag;
  uint64_t *head_in, *tail_in, *head_out, *tail_out;
  char *fifo_in, *fifo_out;
  uint32_t m_in = 0, m_out = 0;
  uint64_t seen_head = 0, seen_tail = 0;  // lane 0: last values observed

  __device__ RingWarp(const RingArgs& args, int r_, int ch, int warp, int lane_, int W, uint64_t E_,
                      uint32_t tag_)
      : a(args), r(r_), lane(lane_), E(E_), tag(tag_) {
    const int n = a.n;
    prev = (r + n - 1) % n;
    next = (r + 1) % n;
    const size_t link_in = (size_t)prev * a.channels + ch;
    const size_t link_out = (size_t)r * a.channels + ch;
    head_in = a.head + link_in * W + warp;
    tail_in = a.tail + link_in * W + warp;
    head_out = a.head + link_out * W + warp;
    tail_out = a.tail + link_out * W + warp;
    const size_t wregion = (size_t)warp * 32 * UPT * 16 * AW;
    fifo_in = a.fifo + link_in * a.K * a.slot_bytes + wregion;
    fifo_out = a.fifo + link_out * a.K * a.slot_bytes + wregion;
  }

  // Lane 0 waits for the next incoming message and / or a free outgoing
  // slot; the warp learns the outcome.  False: the call was aborted.
  __device__ __forceinline__ bool wait(bool need_in, bool need_out, int step) {
    int ok = 1;
    if (lane == 0) {
      if (need_in) {
        const uint64_t want = E | (uint64_t)(m_in + 1);
        if (seen_head < want) ok = wait_geq(head_in, want, &seen_head, a.wait, tag, r, prev, step);
      }
      if (ok && need_out && m_out >= (uint32_t)a.K) {
        const uint64_t want = E | (uint64_t)(m_out - a.K + 1);
        if (seen_tail < want) ok = wait_geq(tail_out, want, &seen_tail, a.wait, tag, r, next, step);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
  }

  // Publish the message just written and / or free the slot just read.
  __device__ __forceinline__ void post(bool sent, bool consumed) {
    __syncwarp();
    if (lane == 0) {
      fence_acq_rel();
      if (sent) st_relaxed(head_out, E | (uint64_t)(m_out + 1));
      if (consumed) st_relaxed(tail_in, E | (uint64_t)(m_in + 1));
    }
    if (sent) ++m_out;
    if (consumed) ++m_in;
  }

  __device__ __forceinline__ char* slot_in() const {
    return fifo_in + (size_t)(m_in % (uint32_t)a.K) * a.slot_bytes;
  }
  __device__ __forceinline__ char* slot_out() const {
    return fifo_out + (size_t)(m_out % (uint32_t)a.K) * a.slot_bytes;
  }

  // Reduce-scatter send of chunk c (first step: own data; later steps:
  // received partial (+) own data).
  __device__ __forceinline__ bool rs_step(int c, bool first, size_t base, int step) {
    if (!wait(!first, true, step)) return false;
    const char* x = static_cast<const char*>(a.in[r]) + a.ibase[c] * ES;
    char* si = slot_in();
    char* so = slot_out();
    uint4 xv[UPT];
    int v[UPT];
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = base + (size_t)j * 32 + lane;
      v[j] = unit_valid<DT>(u, a.len[c]);
      if (v[j] > 0) xv[j] = load_in<DT, VEC>(x, u, v[j]);
    }
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      const size_t w = (size_t)(j * 32 + lane) * AW;
      Acc s;
      if (first) {
        acc_init<DT>(s, xv[j]);
      } else {
        uint4 p[AW];
#pragma unroll
        for (int q = 0; q < AW; ++q) p[q] = ld_l2(si + (w + q) * 16);
        acc_from_words<DT>(s, p);
        acc_add<DT>(s, xv[j]);
      }
      uint4 o[AW];
      acc_to_words<DT>(s, o);
#pragma unroll
      for (int q = 0; q < AW; ++q) st_l2(so + (w + q) * 16, o[q]);
    }
    post(true, !first);
    return true;
  }

  // Last reduce-scatter step: chunk r is complete; store it, and forward it
  // (as the first all-gather message) when `fwd`.
  __device__ __forceinline__ bool rs_final(size_t base, bool fwd, int step) {
    if (!wait(a.n > 1, fwd, step)) return false;
    const char* x = static_cast<const char*>(a.in[r]) + a.ibase[r] * ES;
    char* y = static_cast<char*>(a.out[r]) + a.obase[r] * ES;
    char* si = slot_in();
    char* so = slot_out();
    uint4 xv[UPT];
    int v[UPT];
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = base + (size_t)j * 32 + lane;
      v[j] = unit_valid<DT>(u, a.len[r]);
      if (v[j] > 0) xv[j] = load_in<DT, VEC>(x, u, v[j]);
    }
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      const size_t u = base + (size_t)j * 32 + lane;
      Acc s;
      if (a.n > 1) {
        uint4 p[AW];
#pragma unroll
        for (int q = 0; q < AW; ++q) p[q] = ld_l2(si + ((size_t)(j * 32 + lane) * AW + q) * 16);
        acc_from_words<DT>(s, p);
        acc_add<DT>(s, xv[j]);
      } else {
        acc_init<DT>(s, xv[j]);
      }
      const uint4 out = acc_narrow<DT>(s);
      store_out<DT, VEC, true>(y, u, v[j], out);
      if (fwd) st_l2(so + (size_t)(j * 32 + lane) * 16, out);
    }
    post(fwd, a.n > 1);
    return true;
  }

  // All-gather start (all-gather mode): the own shard is chunk r.
  __device__ __forceinline__ bool ag_first(size_t base, int step) {
    if (!wait(false, true, step)) return false;
    const char* x = static_cast<const char*>(a.in[r]) + a.ibase[r] * ES;
    char* y = static_cast<char*>(a.out[r]) + a.obase[r] * ES;
    char* so = slot_out();
    uint4 xv[UPT];
    int v[UPT];
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = base + (size_t)j * 32 + lane;
      v[j] = unit_valid<DT>(u, a.len[r]);
      if (v[j] > 0) xv[j] = load_in<DT, VEC>(x, u, v[j]);
    }
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      const size_t u = base + (size_t)j * 32 + lane;
      store_out<DT, VEC, true>(y, u, v[j], xv[j]);
      st_l2(so + (size_t)(j * 32 + lane) * 16, xv[j]);
    }
    post(true, false);
    return true;
  }

  // All-gather step: receive chunk c, store it, forward it unless `last`.
  __device__ __forceinline__ bool ag_step(int c, bool last, size_t base, int step) {
    if (!wait(true, !last, step)) return false;
    char* y = static_cast<char*>(a.out[r]) + a.obase[c] * ES;
    char* si = slot_in();
    char* so = slot_out();
    uint4 yv[UPT];
    int v[UPT];
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = base + (size_t)j * 32 + lane;
      v[j] = unit_valid<DT>(u, a.len[c]);
      if (v[j] > 0) yv[j] = ld_l2(si + (size_t)(j * 32 + lane) * 16);
    }
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      const size_t u = base + (size_t)j * 32 + lane;
      store_out<DT, VEC, true>(y, u, v[j], yv[j]);
      if (!last) st_l2(so + (size_t)(j * 32 + lane) * 16, yv[j]);
    }
    post(!last, true);
    return true;
  }

  __device__ void run(int ch, int warp) {
    const int n = a.n, C = a.channels, G = a.G;
    const size_t slice = (size_t)a.slice_units;
    size_t maxu = 0;
    for (int c = 0; c < n; ++c) {
      const size_t u = (a.len[c] + PU - 1) / PU;
      maxu = u > maxu ? u : maxu;
    }
    const size_t per_iter = (size_t)C * G * slice;
    const size_t iters = (maxu + per_iter - 1) / per_iter;
    const size_t wofs = (size_t)warp * 32 * UPT;
    for (size_t it = 0; it < iters; ++it) {
      const size_t it_base = (it * C + ch) * G * slice + wofs;
      int step = 0;
      if (a.mode != kRingAllGather) {
        for (int s = 0; s + 1 < n; ++s, ++step) {
          const int c = ((r - s - 1) % n + n) % n;
          for (int g = 0; g < G; ++g)
            if (!rs_step(c, s == 0, it_base + (size_t)g * slice, step)) return;
        }
        const bool fwd = a.mode == kRingAllReduce && n > 1;
        for (int g = 0; g < G; ++g)
          if (!rs_final(it_base + (size_t)g * slice, fwd, step)) return;
        ++step;
        if (a.mode == kRingReduceScatter || n == 1) continue;
      } else {
        for (int g = 0; g < G; ++g)
          if (!ag_first(it_base + (size_t)g * slice, step)) return;
        ++step;
      }
      // all-gather steps 1 .. n-1: receive chunk (r - s) mod n
      for (int s = 1; s < n; ++s, ++step) {
        const int c = ((r - s) % n + n) % n;
        const bool last = s == n - 1;
        for (int g = 0; g < G; ++g)
          if (!ag_step(c, last, it_base + (size_t)g * slice, step)) return;
      }
    }
  }
};

template <int DT, bool VEC>
__global__ void __launch_bounds__(kRingThreads) ring_kernel(const __grid_constant__ RingArgs a) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch;
  const int r = blockIdx.x % a.n, ch = blockIdx.x / a.n;
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (r != a.wait.skip_rank) {
    RingWarp<DT, VEC> w(a, r, ch, warp, lane, W, (uint64_t)epoch << 32, epoch + 1u);
    w.run(ch, warp);
  }
  arrive_end(a.wait.sync, epoch);
}

template <int DT, bool VEC>
static const void* ring_fn() {
  return reinterpret_cast<const void*>(&ring_kernel<DT, VEC>);
}

static const void* ring_pick(int dt, bool vec) {
  if (dt == RRA_INT32) return vec ? ring_fn<RRA_INT32, true>() : ring_fn<RRA_INT32, false>();
  if (dt == RRA_FLOAT32) return vec ? ring_fn<RRA_FLOAT32, true>() : ring_fn<RRA_FLOAT32, false>();
  if (dt == RRA_BFLOAT16) return vec ? ring_fn<RRA_BFLOAT16, true>() : ring_fn<RRA_BFLOAT16, false>();
  return nullptr;
}

cudaError_t ring_occupancy(int dt, bool vec, int* max_blocks_per_sm) {
  const void* f = ring_pick(dt, vec);
  if (!f) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, f, kRingThreads, 0);
}

cudaError_t launch_ring(int dt, bool vec, const RingArgs& a, int grid, cudaStream_t s) {
  const void* f = ring_pick(dt, vec);
  if (!f) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRingThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<RingArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace rra
