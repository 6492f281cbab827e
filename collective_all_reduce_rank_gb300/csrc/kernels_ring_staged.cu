// kernels_ring_staged.cu -- the ring (Simple protocol) with whole-CTA
// messages staged in shared memory by bulk copies.
//
// Same schedule and summation order as kernels_ring.cu ("NCCL collectives,
// ring all-reduce & launching TP/PP", sections "Direct answer" and "Deep
// dive"; "Collective communication: NCCL's algorithms and protocols...",
// sections "Algorithms" and "Protocols"): reduce-scatter step s sends the
// partial of chunk (r-s-1) to r+1, which adds its own slice; chunk c ends
// summed x_{c+1}, ..., x_{c-1}, x_c; the all-gather forwards the reduced
// chunks.  Simple protocol: the sender writes a message, fences, and raises
// a counter the receiver acquires before it reads.
//
// One persistent cooperative launch of n x C CTAs; CTA (r, ch) is channel ch
// of virtual rank r and owns link (r -> r+1, ch): a FIFO of K message slots
// in the workspace (kept in L2) with a head counter (messages posted) and a
// tail counter (messages consumed, i.e. credits).  A message is a tile of T
// 16-byte input units.  The CTA runs a pipeline over D shared-memory stages
// with warp roles:
//   warp 0 (X loader): bulk-copies the rank's own input tile of message q
//     into stage q mod D (it never waits on a peer, so HBM reads run ahead);
//   warps 1..P (P loaders, message q taken by warp 1 + q mod P): acquire
//     the incoming head counter and the outgoing tail counter side by side,
//     then bulk-copy the incoming message into the stage.  Each acquire is an
//     L2 round trip; P warps keep P of them in flight.  At most D of them
//     work: a loader tests the "stage free" mbarrier by phase parity, which
//     is only sound while it cannot be 2D messages ahead of the consumers,
//     and a loader's previous message (P earlier) bounds that lead to
//     P + D <= 2D;
//   warps P+2.. (consumers): wait for both copies, add, write the outgoing
//     slot or the output, release the stage, publish "message q done";
//   warp P+1 (signaller): once every consumer warp has finished a run of
//     messages, one fence then one head update for all of them, so the
//     fence latency is paid once per batch and never stalls a consumer.
// Each step sends G messages, so the message a rank needs next was posted G
// messages earlier and the hop latency hides behind the other G-1.
// Reduce-scatter partials travel through the FIFO slots; a value already in
// the element type (the finished chunk, and every all-gather forward) is
// not copied into a slot: the sender stores it in its own output, kept in
// L2, and posts it, and the receiver bulk-copies it from there (an output is
// never rewritten within a call, so these messages need no credit).  The
// first reduce-scatter message is no partial at all, only the sender's own
// input tile: the receiver bulk-copies it from the sender's input at its
// step 1, with no wait, and the sender skips step 0.  So of the 2(n-1)
// sends per rank only n-2 go through slots, and L2 bandwidth is what bounds
// this ring.  Only the inputs are read from HBM (each once, by the sender
// or, for the first message, by its receiver) and only the outputs written
// to it.  Two P loaders and twelve consumers make a CTA of 16 warps, which
// caps a thread at 128 registers (the consumers' batches are sized to fit
// without spilling); at the default tiles only two or three stages fit.  Every
// role walks the message sequence with counters (no integer division on
// the per-message path), and every mbarrier wait suspends the warp in
// hardware rather than spinning, so waiting roles leave the issue slots to
// the consumers.
//
// Needs 16-byte aligned buffers and chunk starts.  A chunk's partial last
// 16-byte unit is read and written element-wise by the consumers.  Every
// wait is bounded; on expiry or abort the CTA records the error, waits for
// its own copies in flight and leaves.
#include "staged.cuh"

namespace rra {

constexpr int kStagedPLoaders = 2;
constexpr int kStagedConsumers = 12;
constexpr int kStagedSignaller = 1 + kStagedPLoaders;  // warp index
constexpr int kStagedFirstConsumer = kStagedSignaller + 1;
constexpr int kStagedThreads = (kStagedFirstConsumer + kStagedConsumers) * 32;
constexpr int kStagedMaxStages = 8;

// Position in the message sequence: iteration, step within it (from
// `first`, see staged_first_step), slice g.
struct StagedCursor {
  uint32_t it = 0, step, g = 0, first;
  __device__ __forceinline__ explicit StagedCursor(uint32_t first_) : step(first_), first(first_) {}
  __device__ __forceinline__ void next(int G, int steps) {
    if (++g == (uint32_t)G) {
      g = 0;
      if (++step == (uint32_t)steps) {
        step = first;
        ++it;
      }
    }
  }
};

// The first reduce-scatter step only forwards the sender's own input: its
// receiver reads that tile from the sender's input buffer at the next step
// (a "pulled" message that needs no wait), so a rank's sequence starts at
// step 1 whenever there is a reduce-scatter with two ranks or more.
__host__ __device__ __forceinline__ int staged_first_step(int mode, int n) {
  return mode != kRingAllGather && n >= 2 ? 1 : 0;
}

struct StagedMsg {
  int c;           // chunk
  bool x;          // reads the rank's own input tile
  bool in;         // receives a message (pulled from the sender's output when !x)
  bool pin;        // the incoming message is the sender's input tile (step 1)
  bool send;       // sends a message (posted in its own output when store)
  bool store;      // writes the output
  int nw;          // 16-byte words per unit in the incoming message
  size_t base;     // first unit of the tile inside chunk c
  uint32_t units;  // units of the tile with at least one valid element
  uint32_t xfull;  // units of the tile with all elements valid
};

template <int DT>
__device__ __forceinline__ StagedMsg staged_msg(const RingArgs& a, int r, int ch, const StagedCursor& k) {
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int AW = Elem<DT>::kAccWords;
  const int n = a.n, step = (int)k.step;
  StagedMsg m;
  m.base = (((size_t)k.it * a.channels + ch) * a.G + k.g) * (size_t)a.slice_units;
  int c;
  m.pin = false;
  if (a.mode != kRingAllGather) {
    if (step < n - 1) {  // reduce-scatter step s = step (>= 1: step 0 is pulled)
      c = r - step - 1;
      m.x = true;
      m.in = step > 0;
      m.pin = step == 1;
      m.send = true;
      m.store = false;
      m.nw = step == 1 ? 1 : AW;
    } else if (step == n - 1) {  // last reduce-scatter step: chunk r complete
      c = r;
      m.x = true;
      m.in = n > 1;
      m.pin = n == 2;
      m.send = a.mode == kRingAllReduce && n > 1;
      m.store = true;
      m.nw = n == 2 ? 1 : AW;
    } else {  // all-gather step s
      const int s = step - (n - 1);
      c = r - s;
      m.x = false;
      m.in = true;
      m.send = s < n - 1;
      m.store = true;
      m.nw = 1;
    }
  } else {
    c = r - step;
    m.x = step == 0;
    m.in = step > 0;
    m.send = step < n - 1;
    m.store = true;
    m.nw = 1;
  }
  m.c = c < 0 ? c + n : c;
  const size_t len = a.len[m.c];
  const size_t total = (len + PU - 1) / PU, whole = len / PU;
  const size_t T = (size_t)a.slice_units;
  m.units = m.base < total ? (uint32_t)(total - m.base < T ? total - m.base : T) : 0u;
  m.xfull = m.base < whole ? (uint32_t)(whole - m.base < T ? whole - m.base : T) : 0u;
  return m;
}

struct StagedShared {
  uint64_t fullx[kStagedMaxStages];
  uint64_t fullp[kStagedMaxStages];
  uint64_t empty[kStagedMaxStages];
  uint32_t done[kStagedConsumers];  // messages finished by each consumer warp
  uint32_t abort;
  uint32_t epoch;
};

// Consumer fast paths over whole units.  Thread unit k of a batch is
// u0 + k * (consumer threads), so each warp access is 512 contiguous bytes.
// Batch: units a thread loads before it adds (bfloat16 holds two
// accumulator words per unit, so half as many).  Twelve consumer warps with
// batches of 2 (bfloat16 1) measured faster on GB300 than eight with 4 (2):
// 8 x 100 MB fp32 all-reduce 0.675 -> 0.693 of the HBM copy rate,
// reduce-scatter 0.676 -> 0.691, all-gather 0.701 -> 0.745, bf16 8 x 50M
// 0.482 -> 0.488; 10, 14 and 16 consumers, and batches of 1 or 3, measured
// between the two or slower.
template <int DT>
__host__ __device__ constexpr int staged_batch() {
  return Elem<DT>::kAccWords == 2 ? 1 : 2;
}
constexpr int kStagedNT = kStagedConsumers * 32;

// reduce-scatter step: partial (+ incoming partial) -> outgoing slot, as
// accumulator words
// The incoming message of unit u: accumulator words (a partial from a
// slot), or the element type (the sender's input tile, `pin`).  For 4-byte
// types the two are the same bits, so only bfloat16 tells them apart.
template <int DT>
__device__ __forceinline__ void staged_load_in(const unsigned char* ps, uint32_t u, bool pin, uint4* w) {
  constexpr int AW = Elem<DT>::kAccWords;
  if (AW == 2 && pin) {
    w[0] = lds128(ps + (size_t)u * 16);
  } else {
#pragma unroll
    for (int q = 0; q < AW; ++q) w[q] = lds128(ps + ((size_t)u * AW + q) * 16);
  }
}

// s = incoming (+) x, in that order
template <int DT>
__device__ __forceinline__ void staged_acc_in(Acc& s, const uint4* w, bool pin, uint4 x) {
  if (Elem<DT>::kAccWords == 2 && pin)
    acc_init<DT>(s, w[0]);  // the sender's own slice
  else
    acc_from_words<DT>(s, w);  // the partial so far
  acc_add<DT>(s, x);           // then this rank's slice
}

template <int DT>
__device__ __forceinline__ void staged_partial(const unsigned char* xs, const unsigned char* ps, char* so,
                                               uint32_t u0, uint32_t units, bool in, bool pin) {
  constexpr int AW = Elem<DT>::kAccWords;
  constexpr int B = staged_batch<DT>();
  uint4 xv[B], pw[B][AW];
#pragma unroll
  for (int k = 0; k < B; ++k) {
    const uint32_t u = u0 + k * kStagedNT;
    if (u < units) {
      xv[k] = lds128(xs + (size_t)u * 16);
      if (in) staged_load_in<DT>(ps, u, pin, pw[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < B; ++k) {
    const uint32_t u = u0 + k * kStagedNT;
    if (u < units) {
      Acc s;
      if (in)
        staged_acc_in<DT>(s, pw[k], pin, xv[k]);
      else
        acc_init<DT>(s, xv[k]);
      uint4 o[2];
      acc_to_words<DT>(s, o);
#pragma unroll
      for (int q = 0; q < AW; ++q) st_l2(so + ((size_t)u * AW + q) * 16, o[q]);
    }
  }
}

// last reduce-scatter step (or the all-gather's own shard): the value in
// the element type -> output (posted to the successor when sending)
template <int DT>
__device__ __forceinline__ void staged_final(const unsigned char* xs, const unsigned char* ps, char* yg,
                                             size_t base, uint32_t u0, uint32_t units, bool in, bool pin,
                                             bool send) {
  constexpr int AW = Elem<DT>::kAccWords;
  constexpr int B = staged_batch<DT>();
  uint4 xv[B], pw[B][AW];
#pragma unroll
  for (int k = 0; k < B; ++k) {
    const uint32_t u = u0 + k * kStagedNT;
    if (u < units) {
      xv[k] = lds128(xs + (size_t)u * 16);
      if (in) staged_load_in<DT>(ps, u, pin, pw[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < B; ++k) {
    const uint32_t u = u0 + k * kStagedNT;
    if (u < units) {
      Acc s;
      if (in)
        staged_acc_in<DT>(s, pw[k], pin, xv[k]);
      else
        acc_init<DT>(s, xv[k]);
      const uint4 val = acc_narrow<DT>(s);
      // a posted value stays in L2 for the successor's read
      if (send)
        st_l2(yg + (base + u) * 16, val);
      else
        st_stream(yg + (base + u) * 16, val);
    }
  }
}

// all-gather step: incoming value -> output (posted to the successor when
// sending)
template <int DT>
__device__ __forceinline__ void staged_forward(const unsigned char* ps, char* yg, size_t base, uint32_t u0,
                                               uint32_t units, bool send) {
  constexpr int B = staged_batch<DT>();
  uint4 v[B];
#pragma unroll
  for (int k = 0; k < B; ++k) {
    const uint32_t u = u0 + k * kStagedNT;
    if (u < units) v[k] = lds128(ps + (size_t)u * 16);
  }
#pragma unroll
  for (int k = 0; k < B; ++k) {
    const uint32_t u = u0 + k * kStagedNT;
    if (u < units) {
      if (send)
        st_l2(yg + (base + u) * 16, v[k]);
      else
        st_stream(yg + (base + u) * 16, v[k]);
    }
  }
}

// A tile with a partial last unit (the end of a ragged chunk): one unit per
// thread at a time, element-wise where the unit is partial.
template <int DT>
__device__ __forceinline__ void staged_ragged(const StagedMsg& m, const unsigned char* xs, const unsigned char* ps,
                                              char* so, const char* xg, const char* pg, const char* pxg, char* yg,
                                              size_t len, int tid) {
  constexpr int AW = Elem<DT>::kAccWords;
  for (uint32_t u = tid; u < m.units; u += kStagedNT) {
    const size_t gu = m.base + u;
    const int v = unit_valid<DT>(gu, len);
    if (!m.x) {
      // all-gather step: the value, in the element type, from the sender's
      // output (its partial last unit read directly)
      const uint4 val = u < m.xfull ? lds128(ps + (size_t)u * 16) : ld_partial_l2<DT>(pg + gu * 16, v);
      if (m.send)
        store_out<DT, true, false>(yg, gu, v, val);
      else
        store_out<DT, true, true>(yg, gu, v, val);
      continue;
    }
    const uint4 xv = u < m.xfull ? lds128(xs + (size_t)u * 16) : ld_partial<DT>(xg + gu * 16, v);
    Acc s;
    if (m.pin) {
      // the sender's input tile (its partial last unit read directly)
      const uint4 w = u < m.xfull ? lds128(ps + (size_t)u * 16) : ld_partial<DT>(pxg + gu * 16, v);
      staged_acc_in<DT>(s, &w, true, xv);
    } else if (m.in) {
      uint4 w[2];
      w[0] = lds128(ps + (size_t)u * 16 * AW);
      if (AW == 2) w[1] = lds128(ps + (size_t)u * 16 * AW + 16);
      staged_acc_in<DT>(s, w, false, xv);
    } else {
      acc_init<DT>(s, xv);
    }
    if (!m.store) {
      uint4 o[2];
      acc_to_words<DT>(s, o);
      st_l2(so + (size_t)u * 16 * AW, o[0]);
      if (AW == 2) st_l2(so + (size_t)u * 16 * AW + 16, o[1]);
    } else {
      const uint4 val = acc_narrow<DT>(s);
      if (m.send)
        store_out<DT, true, false>(yg, gu, v, val);
      else
        store_out<DT, true, true>(yg, gu, v, val);
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kStagedThreads, 1) ring_staged_kernel(const __grid_constant__ RingArgs a) {
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int ES = Elem<DT>::kSize;
  constexpr int AW = Elem<DT>::kAccWords;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ StagedShared sh;
  const int n = a.n, C = a.channels, G = a.G, K = a.K, D = a.stages;
  const int T = a.slice_units;
  const int r = blockIdx.x % n, ch = blockIdx.x / n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t xstage = (size_t)T * 16, pstage = (size_t)T * 16 * AW;
  unsigned char* xbuf = smem;                       // [D][T] units
  unsigned char* pbuf = smem + (size_t)D * xstage;  // [D][T * AW] words

  if (threadIdx.x == 0) {
    sh.epoch = read_epoch(a.wait.sync);
    sh.abort = 0;
    for (int b = 0; b < D; ++b) {
      c_mbar_init(&sh.fullx[b], 1);
      c_mbar_init(&sh.fullp[b], 1);
      c_mbar_init(&sh.empty[b], kStagedConsumers);
    }
    for (int w = 0; w < kStagedConsumers; ++w) sh.done[w] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint32_t epoch = sh.epoch;
  const uint64_t E = (uint64_t)epoch << 32;
  const uint32_t tag = epoch + 1u;
  volatile uint32_t* abort = &sh.abort;

  size_t maxu = 0;
  for (int c = 0; c < n; ++c) {
    const size_t u = (a.len[c] + PU - 1) / PU;
    maxu = u > maxu ? u : maxu;
  }
  const int steps = a.mode == kRingAllReduce ? 2 * n - 1 : n;
  const uint32_t first = (uint32_t)staged_first_step(a.mode, n);
  const size_t per_iter_units = (size_t)C * G * T;
  // messages per CTA (the host keeps this below 2^31)
  const uint32_t Q =
      (uint32_t)((maxu + per_iter_units - 1) / per_iter_units) * (uint32_t)((steps - (int)first) * G);

  const int prev = (r + n - 1) % n, next = (r + 1) % n;
  const size_t link_in = (size_t)prev * C + ch, link_out = (size_t)r * C + ch;
  uint64_t* head_in = a.head + link_in;
  uint64_t* tail_in = a.tail + link_in;
  uint64_t* head_out = a.head + link_out;
  uint64_t* tail_out = a.tail + link_out;
  char* fifo_in = a.fifo + link_in * (size_t)K * a.slot_bytes;
  char* fifo_out = a.fifo + link_out * (size_t)K * a.slot_bytes;
  const bool active = r != a.wait.skip_rank;

  if (active && warp <= kStagedPLoaders) {
    // ---------------- loaders: warp 0 the own input, warps 1..P the incoming slots ----------------
    const bool px = warp == 0;
    const uint32_t np = (uint32_t)min(kStagedPLoaders, D);  // P loaders at work
    const uint32_t mine = px ? 0u : (uint32_t)(warp - 1);  // P loader: messages q = mine mod np
    uint32_t pos = 0;                                       // q mod np
    uint64_t* full = px ? sh.fullx : sh.fullp;
    StagedCursor k(first);
    StagedStage st;
    // m_in: messages received (head counter); s_in / s_out: partials
    // received / sent through slots (slot index, credits)
    uint32_t m_in = 0, s_in = 0, s_out = 0, slot_in = 0;
    uint64_t seen_head = 0, seen_tail = 0;
    uint32_t q = 0;
    if (mine >= np) q = Q;  // idle P loader
    for (; q < Q; ++q, k.next(G, steps), st.next(D), pos = pos + 1 == np ? 0u : pos + 1) {
      const StagedMsg m = staged_msg<DT>(a, r, ch, k);
      const bool posted = m.in && !m.pin;  // counted on the head counter
      const bool slot_recv = posted && m.x, slot_send = m.send && !m.store;
      if (!px && pos != mine) {  // another P loader's message: only count it
        if (posted) ++m_in;
        if (slot_recv) {
          ++s_in;
          if (++slot_in == (uint32_t)K) slot_in = 0;
        }
        if (slot_send) ++s_out;
        continue;
      }
      int ok = 1;
      if (lane == 0 && q >= (uint32_t)D && !staged_mbar_wait(&sh.empty[st.b], st.ph ^ 1u, abort, a.wait.timeout_ns)) {
        if (!*abort) record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, (int)q, tag);
        ok = 0;
      }
      if (!px) {
        // incoming message posted, and a free outgoing slot, side by side
        if (ok && posted && lane == 0) {
          const uint64_t want = E | (uint64_t)(m_in + 1);
          if (seen_head < want) ok = wait_geq(head_in, want, &seen_head, a.wait, tag, r, prev, (int)q);
        }
        if (slot_send && lane == 1 && s_out >= (uint32_t)K) {
          const uint64_t want = E | (uint64_t)(s_out - K + 1);
          if (seen_tail < want) ok = wait_geq(tail_out, want, &seen_tail, a.wait, tag, r, next, (int)q);
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        if (px) {
          const uint32_t bytes = m.x ? m.xfull * 16u : 0u;
          c_mbar_arrive_tx(&full[st.b], bytes);
          if (bytes)
            bulk_load_stream(xbuf + (size_t)st.b * xstage,
                             static_cast<const char*>(a.in[r]) + (a.ibase[m.c] + m.base * PU) * ES, bytes, &full[st.b]);
        } else {
          // a partial from the slot, or whole units of the sender's output
          // (a value) or of its input (the first partial)
          const uint32_t bytes = !m.in ? 0u : (slot_recv ? m.units * 16u * (uint32_t)m.nw : m.xfull * 16u);
          if (bytes && posted) fence_proxy_async_global();  // generic-proxy writes acquired above, read by the async proxy
          c_mbar_arrive_tx(&full[st.b], bytes);
          if (bytes && slot_recv)
            c_bulk_load(pbuf + (size_t)st.b * pstage, fifo_in + (size_t)slot_in * a.slot_bytes, bytes, &full[st.b]);
          else if (bytes && m.pin)
            bulk_load_stream(pbuf + (size_t)st.b * pstage,
                             static_cast<const char*>(a.in[prev]) + (a.ibase[m.c] + m.base * PU) * ES, bytes,
                             &full[st.b]);
          else if (bytes)
            c_bulk_load(pbuf + (size_t)st.b * pstage,
                        static_cast<const char*>(a.out[prev]) + (a.obase[m.c] + m.base * PU) * ES, bytes, &full[st.b]);
        }
      }
      if (posted) ++m_in;
      if (slot_recv) {
        ++s_in;
        if (++slot_in == (uint32_t)K) slot_in = 0;
      }
      if (slot_send) ++s_out;
    }
    if (q < Q && lane == 0) {
      *abort = 1;
      // copies this warp issued that nobody will consume: let them land
      // (the last D messages, each the latest use of its stage)
      StagedStage w;
      const uint32_t lo = q > (uint32_t)D ? q - D : 0;
      for (uint32_t j = 0; j < q; ++j, w.next(D))
        if (j >= lo && (px || j % np == mine)) c_mbar_wait(&full[w.b], w.ph, a.wait.timeout_ns);
    }
  } else if (active && warp == kStagedSignaller) {
    // ---------------- signaller ----------------
    StagedCursor k(first);
    uint32_t q = 0;  // messages published
    uint32_t m_out = 0;
    uint64_t t0 = 0;
    uint32_t spins = 0;
    while (q < Q) {
      uint32_t d = 0xffffffffu;
      if (lane < kStagedConsumers) d = ld_acquire_cta_u32(&sh.done[lane]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d = min(d, __shfl_xor_sync(0xffffffffu, d, o));
      if (d > q) {
        uint32_t sends = 0;
        for (; q < d; ++q, k.next(G, steps)) sends += staged_msg<DT>(a, r, ch, k).send ? 1u : 0u;
        if (sends && lane == 0) {
          fence_acq_rel();
          red_max_relaxed(head_out, E | (uint64_t)(m_out + sends));
        }
        m_out += sends;
        spins = 0;
        continue;
      }
      if (spins == 0) t0 = globaltimer();
      ++spins;
      int stop = 0;
      if (lane == 0 && (spins & 31u) == 0u &&
          (*abort || globaltimer() - t0 > 2 * a.wait.timeout_ns || spins >= kMaxSpin)) {
        if (!*abort) {
          record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, (int)q, tag);
          *abort = 1;
        }
        stop = 1;
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;
      __nanosleep(spins < 8 ? 32 : 128);  // a poll of shared memory; keep its issue slots few
    }
  } else if (active && warp >= kStagedFirstConsumer) {
    // ---------------- consumers ----------------
    const int cw = warp - kStagedFirstConsumer;
    const int tid = cw * 32 + lane;
    StagedCursor k(first);
    StagedStage st;
    uint32_t s_in = 0, slot_out = 0;  // partials received; next outgoing slot
    for (uint32_t q = 0; q < Q; ++q, k.next(G, steps), st.next(D)) {
      const StagedMsg m = staged_msg<DT>(a, r, ch, k);
      const bool slot_recv = m.in && !m.pin && m.x, slot_send = m.send && !m.store;
      int ok = 1;
      if (lane == 0 && !(staged_mbar_wait(&sh.fullx[st.b], st.ph, abort, a.wait.timeout_ns) &&
                         staged_mbar_wait(&sh.fullp[st.b], st.ph, abort, a.wait.timeout_ns))) {
        if (!*abort) record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, (int)q, tag);
        ok = 0;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) *abort = 1;
        break;
      }
      // every lane reads the stage: make the completed copies visible to it
      mbar_try_cta(&sh.fullx[st.b], st.ph);
      mbar_try_cta(&sh.fullp[st.b], st.ph);
      if (slot_recv && tid == 0) red_max_relaxed(tail_in, E | (uint64_t)(s_in + 1));  // slot copied out: credit
      const unsigned char* xs = xbuf + (size_t)st.b * xstage;
      const unsigned char* ps = pbuf + (size_t)st.b * pstage;
      char* so = fifo_out + (size_t)slot_out * a.slot_bytes;
      char* yg = static_cast<char*>(a.out[r]) + a.obase[m.c] * ES;
      if (m.units == m.xfull) {
        // every unit whole: each thread loads its batch of units from the
        // stage first, then adds, then stores
        for (uint32_t u0 = tid; u0 < m.units; u0 += kStagedNT * staged_batch<DT>()) {
          if (!m.x)
            staged_forward<DT>(ps, yg, m.base, u0, m.units, m.send);
          else if (!m.store)
            staged_partial<DT>(xs, ps, so, u0, m.units, m.in, m.pin);
          else
            staged_final<DT>(xs, ps, yg, m.base, u0, m.units, m.in, m.pin, m.send);
        }
      } else {
        staged_ragged<DT>(m, xs, ps, so, static_cast<const char*>(a.in[r]) + a.ibase[m.c] * ES,
                          static_cast<const char*>(a.out[prev]) + a.obase[m.c] * ES,
                          static_cast<const char*>(a.in[prev]) + a.ibase[m.c] * ES, yg, a.len[m.c], tid);
      }
      __syncwarp();
      if (lane == 0) {
        c_mbar_arrive_tx(&sh.empty[st.b], 0);  // this warp no longer reads the stage
        st_release_cta_u32(&sh.done[cw], q + 1);
      }
      if (slot_recv) ++s_in;
      if (slot_send && ++slot_out == (uint32_t)K) slot_out = 0;
    }
  }
  arrive_end(a.wait.sync, epoch);
}

template <int DT>
static const void* staged_fn() {
  return reinterpret_cast<const void*>(&ring_staged_kernel<DT>);
}

static const void* staged_pick(int dt) {
  if (dt == RRA_INT32) return staged_fn<RRA_INT32>();
  if (dt == RRA_FLOAT32) return staged_fn<RRA_FLOAT32>();
  if (dt == RRA_BFLOAT16) return staged_fn<RRA_BFLOAT16>();
  return nullptr;
}

size_t ring_staged_smem(int dt, int tile_units, int stages) {
  const size_t aw = dt == RRA_BFLOAT16 ? 2 : 1;
  return (size_t)stages * (size_t)tile_units * 16 * (1 + aw);
}

cudaError_t ring_staged_occupancy(int dt, int tile_units, int stages, int* max_blocks_per_sm) {
  const void* f = staged_pick(dt);
  if (!f || stages < 1 || stages > kStagedMaxStages) return cudaErrorInvalidValue;
  const size_t smem = ring_staged_smem(dt, tile_units, stages);
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, f, kStagedThreads, smem);
}

cudaError_t launch_ring_staged(int dt, const RingArgs& a, int grid, cudaStream_t s) {
  const void* f = staged_pick(dt);
  if (!f || a.stages < 1 || a.stages > kStagedMaxStages) return cudaErrorInvalidValue;
  const size_t smem = ring_staged_smem(dt, a.slice_units, a.stages);
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStagedThreads);
  cfg.dynamicSmemBytes = smem;
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
