// kernels_ring.cu -- ring all-reduce and its reduce-scatter / all-gather
// halves, with the Simple or the LL protocol on the ring's links.
//
// "NCCL collectives, ring all-reduce & launching TP/PP", sections "Direct
// answer" and "Deep dive": ring all-reduce = reduce-scatter + all-gather;
// the ring pipelines the data in N chunks so every link is busy.
// "Collective communication: NCCL's algorithms and protocols...", section
// "Algorithms": n-1 reduce-scatter steps and n-1 all-gather steps, each
// GPU sending and receiving 2(n-1)/n S; section "Protocols": LL lines carry
// 4 data bytes and a 4-byte flag that the receiver polls, Simple writes a
// block, fences and then raises a flag.
//
// Schedule, per rank r (indices mod n):
//   RS step s = 0..n-2: send the partial of chunk (r-s-1) to r+1; the
//     receiver adds its own slice of that chunk.  Rank r ends with chunk r,
//     summed x_{r+1}, x_{r+2}, ..., x_{r-1}, x_r.
//   AG step s = 0..n-2: forward chunk (r-s) to r+1, which stores it.
//
// Design on one GPU: one persistent cooperative launch of n x C CTAs; CTA
// (r, ch) is channel ch of virtual rank r and every one of its 16 warps is
// an independent pipeline.  The link r -> r+1 of (channel, warp) is a FIFO
// of K slots in the workspace, small enough to stay in L2.  Each step moves
// G messages (slices); the receiver of slice g in step s+1 needs slice g of
// step s, posted G messages earlier, so latency hides behind the other
// slices.  A sender waits for a free slot on the tail counter the receiver
// raises (credits).
//   Simple: write the slot, __syncwarp, fence, raise the head counter; the
//     receiver acquires the head counter before reading the slot.
//   LL: every 4-byte word travels in an 8-byte line with a flag, written
//     and read as one 64-bit access (single-copy atomic), so no fence and
//     no head counter are needed: the receiver polls the lines themselves.
//     The flag carries the call tag (19 bits, bit 31 set) and the slot's
//     round (12 bits), so a line left from the slot's previous use or an
//     earlier call never matches; the lines live in the workspace's LL
//     region, which holds nothing but LL lines.  Credits are raised once
//     per G messages, and not at all in a call too short to reuse a slot.
// The rank's own input for the next message is loaded before its wait, so
// the HBM latency overlaps the wait.  bfloat16 partial sums travel as
// float32 and are rounded once, at the final reduce-scatter step.  Only the
// inputs are read from HBM and only the outputs written to it.
#include "common.cuh"

namespace rra {

template <int DT, bool VEC, int PROTO>
struct RingWarp {
  static constexpr int PU = Elem<DT>::kPerUnit;
  static constexpr int ES = Elem<DT>::kSize;
  static constexpr int AW = Elem<DT>::kAccWords;
  static constexpr int UPT = ring_units_per_thread(DT, PROTO);
  // bytes a slot reserves per unit (per accumulator word: 16 B Simple, 32 B LL)
  static constexpr int WB = PROTO == kProtoLL ? 32 : 16;

  const RingArgs& a;
  int r, prev, next, lane;
  uint64_t E;
  uint32_t tag;
  uint32_t lin, lout;  // counter index of the incoming and outgoing link (and warp)
  uint32_t m_in = 0, m_out = 0;
  uint64_t seen_head = 0, seen_tail = 0;  // last values observed by the polling lanes
  // Per-message state kept incrementally, so that no step divides by a
  // runtime value (a warp alone on its SM pays the full latency of every
  // dependent instruction, and a division is a chain of dozens): the slot
  // of the next message each way and its index, its LL flag, and the
  // message count modulo G.
  char *sin, *sout;
  uint32_t kin = 0, kout = 0, fin, fout, gin = 0, gout = 0;

  __device__ RingWarp(const RingArgs& args, int r_, int ch, int warp, int lane_, int W, uint64_t E_,
                      uint32_t tag_)
      : a(args), r(r_), lane(lane_), E(E_), tag(tag_) {
    const int n = a.n;
    prev = (r + n - 1) % n;
    next = (r + 1) % n;
    const size_t link_in = (size_t)prev * a.channels + ch;
    const size_t link_out = (size_t)r * a.channels + ch;
    lin = (uint32_t)(link_in * W + warp);
    lout = (uint32_t)(link_out * W + warp);
    const size_t wregion = (size_t)warp * 32 * UPT * AW * WB;
    sin = a.fifo + link_in * a.K * a.slot_bytes + wregion;
    sout = a.fifo + link_out * a.K * a.slot_bytes + wregion;
    fin = fout = ((tag & 0x7FFFFu) | 0x80000u) << 12;
  }

  // LL flag of a message: the slot's round m / K (12 bits) under the call
  // tag (19 bits, top bit always set, so never 0).  A slot can hold lines of
  // any older round -- the messages between may have been empty and never
  // written -- so the round itself must match, not just its parity; the
  // host keeps a call under 4096 rounds per slot.  fin / fout hold the flag
  // of the next message in / out; the round advances when the slot index
  // wraps.
  __device__ __forceinline__ static uint32_t next_round(uint32_t f) { return (f & ~0xFFFu) | ((f + 1u) & 0xFFFu); }

  // Wait for the next incoming message (Simple: lane 0 acquires the head
  // counter) and / or a free outgoing slot (lane 1 acquires the tail
  // counter); the two waits run side by side.  False: the call aborted.
  __device__ __forceinline__ bool wait(bool need_in, bool need_out, int step) {
    int ok = 1;
    // (the out-of-line wait writes the value it saw through a pointer: a
    // copy, so that no pointer into this object escapes and its state stays
    // in registers)
    if (PROTO == kProtoSimple && need_in && lane == 0) {
      const uint64_t want = E | (uint64_t)(m_in + 1);
      if (seen_head < want) {
        uint64_t seen = seen_head;
        ok = wait_geq(a.head + lin, want, &seen, a.wait, tag, r, prev, step);
        seen_head = seen;
      }
    }
    if (need_out && lane == 1 && m_out >= (uint32_t)a.K) {
      const uint64_t want = E | (uint64_t)(m_out - a.K + 1);
      if (seen_tail < want) {
        uint64_t seen = seen_tail;
        ok = wait_geq(a.tail + lout, want, &seen, a.wait, tag, r, next, step);
        seen_tail = seen;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    __syncwarp();
    return ok != 0;
  }

  // Publish the message just written and / or free the slot just read.
  __device__ __forceinline__ void post(bool sent, bool consumed) {
    __syncwarp();
    if (PROTO == kProtoSimple) {
      if (lane == 0) {
        fence_acq_rel();
        if (sent) st_relaxed(a.head + lout, E | (uint64_t)(m_out + 1));
        if (consumed) st_relaxed(a.tail + lin, E | (uint64_t)(m_in + 1));
      }
    } else if (lane == 0) {
      // a credit is a release (the slot's lines were read before it); a
      // call too short to reuse any slot needs none, which takes the
      // release off every hop of a small message
      if (consumed && !a.no_credits && gin + 1 == (uint32_t)a.G) st_release(a.tail + lin, E | (uint64_t)(m_in + 1));
      // progress marker only (the lines carry their own flags): lets a peer
      // that gives up tell a rank that never sent from one stuck behind it
      if (sent && gout + 1 == (uint32_t)a.G) st_relaxed(a.head + lout, E | (uint64_t)(m_out + 1));
    }
    if (sent) {
      ++m_out;
      if (++gout == (uint32_t)a.G) gout = 0;
      sout += a.slot_bytes;
      if (++kout == (uint32_t)a.K) {
        kout = 0;
        sout -= (size_t)a.K * a.slot_bytes;
        fout = next_round(fout);
      }
    }
    if (consumed) {
      ++m_in;
      if (++gin == (uint32_t)a.G) gin = 0;
      sin += a.slot_bytes;
      if (++kin == (uint32_t)a.K) {
        kin = 0;
        sin -= (size_t)a.K * a.slot_bytes;
        fin = next_round(fin);
      }
    }
  }

  __device__ __forceinline__ char* slot_in() const { return sin; }
  __device__ __forceinline__ char* slot_out() const { return sout; }

  // unit j of this lane, word q, in a slot
  __device__ __forceinline__ size_t word_off(int j, int q) const {
    return ((size_t)(j * 32 + lane) * AW + q) * WB;
  }

  __device__ __forceinline__ void put(char* slot, int j, int q, uint4 w) const {
    char* p = slot + word_off(j, q);
    if (PROTO == kProtoSimple) {
      st_l2(p, w);
    } else {
      st_ll_pair(p, fout, w.x, w.y);
      st_ll_pair(p + 16, fout, w.z, w.w);
    }
  }

  // Read the `nw` words of each valid unit of the incoming message.  LL:
  // poll every line until its flag matches (bounded); false on abort.
  __device__ __forceinline__ bool get(const char* slot, const int* v, int nw, uint4 (*w)[2], int step) {
    if (PROTO == kProtoSimple) {
#pragma unroll
      for (int j = 0; j < UPT; ++j)
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (q < nw && v[j] > 0) w[j][q] = ld_l2(slot + word_off(j, q));
      return true;
    }
    const uint32_t f = fin;
    bool done = false;
    uint64_t t0 = 0;
    int ok = 1;
    for (uint32_t it = 0;; ++it) {
      if (!done) {
        bool all = true;
#pragma unroll
        for (int j = 0; j < UPT; ++j)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (q >= nw || v[j] == 0) continue;
            unsigned long long l0, l1, l2, l3;
            const char* p = slot + word_off(j, q);
            ld_ll_pair(p, l0, l1);
            ld_ll_pair(p + 16, l2, l3);
            all = all && (uint32_t)(l0 >> 32) == f && (uint32_t)(l1 >> 32) == f &&
                  (uint32_t)(l2 >> 32) == f && (uint32_t)(l3 >> 32) == f;
            w[j][q] = make_uint4((uint32_t)l0, (uint32_t)l1, (uint32_t)l2, (uint32_t)l3);
          }
        done = all;
      }
      if (__all_sync(0xffffffffu, done)) break;
      if (it == 0) t0 = globaltimer();
      int give_up = 0;
      if ((it & 15u) == 15u && lane == 0) {
        if (aborted(a.wait.status, tag)) {
          give_up = 1;
        } else if (globaltimer() - t0 > a.wait.timeout_ns || it >= kMaxSpin) {
          const bool root = (ld_acquire(a.head + lin) >> 32) != (E >> 32);  // prev sent nothing
          record_error(a.wait.status, RRA_ERR_TIMEOUT, r, prev, step, tag, root);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) {
        ok = 0;
        break;
      }
      if (!done) __nanosleep(32);
    }
    return ok != 0;
  }

  __device__ __forceinline__ void load_x(int c, size_t base, uint4* xv, int* v) const {
    const char* x = static_cast<const char*>(a.in[r]) + a.ibase[c] * ES;
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = base + (size_t)j * 32 + lane;
      v[j] = unit_valid<DT>(u, a.len[c]);
      if (v[j] > 0) xv[j] = load_in<DT, VEC>(x, u, v[j]);
    }
  }

  // The rank's own input for the next message that reads it is loaded one
  // such message ahead, so its HBM latency overlaps the current message.
  // Those messages come in a fixed order: per iteration, the reduce-scatter
  // sends k = 0..n-2 (chunk r-k-1) and the final step (chunk r), G slices
  // each; in all-gather mode only the own shard.
  uint4 xn[UPT];
  int vn[UPT];
  uint32_t xq = 0, xq_total = 0;  // below 2^31, as the message counters
  // where message xq reads the own input: read xk of its iteration (the
  // reduce-scatter's chunk r-xk-1, or chunk r), slice xg, first unit xbase
  int xk = 0, xg = 0;
  size_t xbase = 0;

  __device__ __forceinline__ void prefetch_x() {
    if (xq >= xq_total) return;
    int c = r;
    if (a.mode != kRingAllGather && xk <= a.n - 2) {
      c = r - xk - 1;
      if (c < 0) c += a.n;
    }
    load_x(c, xbase, xn, vn);
  }

  // the next such message: slice g + 1, else the next read, else the next
  // iteration (C x G slices further on)
  __device__ __forceinline__ void advance_x() {
    ++xq;
    const size_t slice = (size_t)a.slice_units;
    xbase += slice;
    if (++xg == a.G) {
      xg = 0;
      xbase -= (size_t)a.G * slice;
      if (++xk == (a.mode == kRingAllGather ? 1 : a.n)) {
        xk = 0;
        xbase += (size_t)a.channels * a.G * slice;
      }
    }
  }

  __device__ __forceinline__ void take_x(uint4* xv, int* v) {
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      xv[j] = xn[j];
      v[j] = vn[j];
    }
    advance_x();
    prefetch_x();
  }

  // Reduce-scatter send of chunk c (first step: own data; later steps:
  // received partial (+) own data).
  __device__ __forceinline__ bool rs_step(int c, bool first, size_t base, int step) {
    uint4 xv[UPT];
    int v[UPT];
    take_x(xv, v);  // chunk c at base, loaded one message ago
    if (!wait(!first, true, step)) return false;
    uint4 p[UPT][2];
    if (!first && !get(slot_in(), v, AW, p, step)) return false;
    char* so = slot_out();
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      Acc s;
      if (first) {
        acc_init<DT>(s, xv[j]);
      } else {
        acc_from_words<DT>(s, p[j]);
        acc_add<DT>(s, xv[j]);
      }
      uint4 o[2];
      acc_to_words<DT>(s, o);
#pragma unroll
      for (int q = 0; q < AW; ++q) put(so, j, q, o[q]);
    }
    post(true, !first);
    return true;
  }

  // Last reduce-scatter step: chunk r is complete; store it, and forward it
  // (as the first all-gather message) when `fwd`.
  __device__ __forceinline__ bool rs_final(size_t base, bool fwd, int step) {
    uint4 xv[UPT];
    int v[UPT];
    take_x(xv, v);  // chunk r at base, loaded one message ago
    if (!wait(a.n > 1, fwd, step)) return false;
    uint4 p[UPT][2];
    if (a.n > 1 && !get(slot_in(), v, AW, p, step)) return false;
    char* y = static_cast<char*>(a.out[r]) + a.obase[r] * ES;
    char* so = slot_out();
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      const size_t u = base + (size_t)j * 32 + lane;
      Acc s;
      if (a.n > 1) {
        acc_from_words<DT>(s, p[j]);
        acc_add<DT>(s, xv[j]);
      } else {
        acc_init<DT>(s, xv[j]);
      }
      const uint4 out = acc_narrow<DT>(s);
      store_out<DT, VEC, true>(y, u, v[j], out);
      if (fwd) put(so, j, 0, out);
    }
    post(fwd, a.n > 1);
    return true;
  }

  // All-gather start (all-gather mode): the own shard is chunk r.
  __device__ __forceinline__ bool ag_first(size_t base, int step) {
    uint4 xv[UPT];
    int v[UPT];
    take_x(xv, v);  // chunk r at base, loaded one message ago
    if (!wait(false, true, step)) return false;
    char* y = static_cast<char*>(a.out[r]) + a.obase[r] * ES;
    char* so = slot_out();
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      const size_t u = base + (size_t)j * 32 + lane;
      store_out<DT, VEC, true>(y, u, v[j], xv[j]);
      put(so, j, 0, xv[j]);
    }
    post(true, false);
    return true;
  }

  // All-gather step: receive chunk c, store it, forward it unless `last`.
  __device__ __forceinline__ bool ag_step(int c, bool last, size_t base, int step) {
    int v[UPT];
#pragma unroll
    for (int j = 0; j < UPT; ++j) v[j] = unit_valid<DT>(base + (size_t)j * 32 + lane, a.len[c]);
    if (!wait(true, !last, step)) return false;
    uint4 p[UPT][2];
    if (!get(slot_in(), v, 1, p, step)) return false;
    char* y = static_cast<char*>(a.out[r]) + a.obase[c] * ES;
    char* so = slot_out();
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      const size_t u = base + (size_t)j * 32 + lane;
      store_out<DT, VEC, true>(y, u, v[j], p[j][0]);
      if (!last) put(so, j, 0, p[j][0]);
    }
    post(!last, true);
    return true;
  }

  __device__ __forceinline__ void run(int ch, int warp) {
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
    xbase = (size_t)ch * G * slice + wofs;
    xq_total = (uint32_t)(iters * (a.mode == kRingAllGather ? 1 : n) * G);
    prefetch_x();
    for (size_t it = 0; it < iters; ++it) {
      const size_t it_base = (it * C + ch) * G * slice + wofs;
      int step = 0;
      if (a.mode != kRingAllGather) {
        for (int s = 0; s + 1 < n; ++s, ++step) {
          const int c = r - s - 1 < 0 ? r - s - 1 + n : r - s - 1;
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
        const int c = r - s < 0 ? r - s + n : r - s;
        const bool last = s == n - 1;
        for (int g = 0; g < G; ++g)
          if (!ag_step(c, last, it_base + (size_t)g * slice, step)) return;
      }
    }
  }
};

template <int DT, bool VEC, int PROTO>
__global__ void __launch_bounds__(kRingThreads, 1) ring_kernel(const __grid_constant__ RingArgs a) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch;
  const int r = blockIdx.x % a.n, ch = blockIdx.x / a.n;
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (r != a.wait.skip_rank) {
    RingWarp<DT, VEC, PROTO> w(a, r, ch, warp, lane, W, (uint64_t)epoch << 32, epoch + 1u);
    w.run(ch, warp);
  }
  arrive_end(a.wait.sync, epoch);
}

template <int DT, bool VEC>
static const void* ring_fn(int proto) {
  return proto == kProtoLL ? reinterpret_cast<const void*>(&ring_kernel<DT, VEC, kProtoLL>)
                           : reinterpret_cast<const void*>(&ring_kernel<DT, VEC, kProtoSimple>);
}

static const void* ring_pick(int dt, bool vec, int proto) {
  if (dt == RRA_INT32) return vec ? ring_fn<RRA_INT32, true>(proto) : ring_fn<RRA_INT32, false>(proto);
  if (dt == RRA_FLOAT32) return vec ? ring_fn<RRA_FLOAT32, true>(proto) : ring_fn<RRA_FLOAT32, false>(proto);
  if (dt == RRA_BFLOAT16) return vec ? ring_fn<RRA_BFLOAT16, true>(proto) : ring_fn<RRA_BFLOAT16, false>(proto);
  return nullptr;
}

cudaError_t ring_occupancy(int dt, bool vec, int proto, int* max_blocks_per_sm) {
  const void* f = ring_pick(dt, vec, proto);
  if (!f) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, f, kRingThreads, 0);
}

cudaError_t launch_ring(int dt, bool vec, int proto, const RingArgs& a, int grid, cudaStream_t s) {
  const void* f = ring_pick(dt, vec, proto);
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
