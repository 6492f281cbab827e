// kernels_tree_staged.cu -- double binary tree all-reduce with whole-CTA
// messages staged in shared memory by bulk copies, links through L2 (the
// machinery of the staged ring, kernels_ring_staged.cu).
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Algorithms": the tree is a
// double binary tree -- reduce up, broadcast down, O(log n) steps, large
// messages pipelined in chunks.  Tree 0 is the binary tree in heap order
// over the ranks (rank r at position r; position p has children 2p+1 and
// 2p+2), tree 1 the same tree over the ranks reversed (rank r at position
// n-1-r).  The message is split in two by the chunk plan for two parts:
// units [0, half_units) go over tree 0, the rest over tree 1.  A node's
// partial is its own data, then its child 2p+1's partial, then its child
// 2p+2's: p = (x (+) p_{2p+1}) (+) p_{2p+2}.  Each root rounds its total
// once and it travels down unchanged, so every rank holds the same bits.
// bfloat16 partials travel as float32.
//
// A rank has children in at most one of the two trees (with n even it is an
// inner node of one and a leaf of the other; with n odd rank (n-1)/2 is a
// leaf of both), so it sends partials up, and posts totals down, in at
// most one tree: its up FIFO, up head and tail and down head are one per
// (rank, channel), as for a single tree.
//
// One persistent cooperative launch of n x C CTAs; CTA (r, ch) is channel
// ch of rank r in BOTH trees, so that every CTA carries one heavy role (the
// tree where the rank has children) and one light one (the tree where it is
// a leaf), and no SM idles behind a leaf's light load.  A leaf's partial is
// its own input, so a leaf sends nothing up: its parent bulk-copies the
// tile from the leaf's input once the leaf has joined the call (the leaf's
// "joined" flag), and the leaf only receives.  Per channel each inner
// non-root node owns an up FIFO (its partials, read by its parent) of K
// slots in the workspace, with a head counter (messages posted) and a tail
// counter (messages the parent has copied out).  The totals going down need
// no FIFO: a node with children stores the total in its own output, kept
// in L2, and posts it on its down head counter; both children bulk-copy it
// from there (an output is written once per call, so these reads need no
// credit).
//
// Message order.  Tiles of T units, G per iteration.  At pipeline time t a
// CTA handles, in this order, the up messages of tile iteration t (in the
// tree where it has children), then the down messages of tile iteration
// t - L of tree 0, then those of tree 1 (the broadcast trails the reduction
// by L iterations, so it overlaps the next L iterations' reduction).
// Every cross-CTA wait is on a message of an earlier time or of the same
// time and kind in the same tree, where up waits run from parent to child
// and down waits from child to parent, so no chain of waits closes on
// itself; a credit wait is on a message at least one time earlier (K >
// G).  Warp roles as in the staged ring: an X loader (bulk-copies the
// node's own input tile), P loaders (acquire the heads of the incoming
// links and the tail of the up link, then bulk-copy the children's slots
// or inputs or the parent's output; at most as many as stages, so the stage
// mbarriers' parity tests stay sound), consumers (add, write the up slot or
// the output), and a signaller (one fence per run of finished messages,
// then the head counters).  Every wait is bounded.
//
// Needs 16-byte aligned buffers.  The last tile's partial 16-byte unit is
// read and written element-wise by the consumers.
#include "staged.cuh"
#include "tree.cuh"

namespace rra {

constexpr int kTreePLoaders = 3;
// Eleven consumers make a CTA of 16 warps (the register cap stays at 128,
// 102-105 used): measured on GB300 against eight, fp32 0.473 -> 0.490 of the
// HBM copy rate at 8 x 100 MB, +1-2% at 2-4 ranks x 256 MiB, bf16 within 1%.
constexpr int kTreeConsumers = 11;
constexpr int kTreeSignaller = 1 + kTreePLoaders;
constexpr int kTreeFirstConsumer = kTreeSignaller + 1;
constexpr int kTreeThreads = (kTreeFirstConsumer + kTreeConsumers) * 32;
constexpr int kTreeMaxStages = 8;
constexpr int kTreeNT = kTreeConsumers * 32;

// The CTA's message classes: 0 = up messages of tree 0, 1 = up messages of
// tree 1, 2 = down messages of tree 0, 3 = down messages of tree 1; class
// c has messages at the times [lo[c], hi[c]) (G per time).
struct TreeSeq {
  uint32_t lo[4], hi[4], tend;
};

// Position in the CTA's message sequence: time t, class, slice g.
struct TreeCursor {
  uint32_t t = 0, cls = 0, g = 0;
  // from (t, cls) on, the first class with messages
  __device__ __forceinline__ void seek(const TreeSeq& s) {
    while (t < s.tend) {
      int found = -1;
#pragma unroll
      for (int c = 3; c >= 0; --c)
        if (c >= (int)cls && s.lo[c] <= t && t < s.hi[c]) found = c;
      if (found >= 0) {
        cls = (uint32_t)found;
        return;
      }
      cls = 0;
      ++t;
    }
  }
  __device__ __forceinline__ explicit TreeCursor(const TreeSeq& s) { seek(s); }
  __device__ __forceinline__ void next(int G, const TreeSeq& s) {
    if (++g < (uint32_t)G) return;
    g = 0;
    ++cls;
    seek(s);
  }
  __device__ __forceinline__ int tree() const { return (int)(cls & 1u); }
  __device__ __forceinline__ bool up() const { return cls < 2u; }
  __device__ __forceinline__ uint32_t tile_it(uint32_t L) const { return cls < 2u ? t : t - L; }
};

struct TreeShared {
  uint64_t fullx[kTreeMaxStages];
  uint64_t fullp[kTreeMaxStages];
  uint64_t empty[kTreeMaxStages];
  uint32_t done[kTreeConsumers];
  uint32_t abort;
  uint32_t epoch;
};

template <int DT>
__global__ void __launch_bounds__(kTreeThreads, 1) tree_staged_kernel(const __grid_constant__ StagedTreeArgs a) {
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int AW = Elem<DT>::kAccWords;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ TreeShared sh;
  const int n = a.n, C = a.channels, G = a.G, K = a.K, D = a.stages, T = a.slice_units;
  const uint32_t L = (uint32_t)a.lag;
  const int r = blockIdx.x % n, ch = blockIdx.x / n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TreeRole R0 = tree_role(0, n, r), R1 = tree_role(1, n, r);
  // the tree where this rank has children (its up messages); with none
  // (n odd, the middle rank) it has down messages only
  const TreeRole Rp = R0.nk > 0 ? R0 : R1;
  const size_t xstage = (size_t)T * 16, pstage = (size_t)T * 16 * AW;
  unsigned char* xbuf = smem;                                 // [D][T] units
  unsigned char* p1buf = smem + (size_t)D * xstage;           // [D][T * AW]: first child / parent
  unsigned char* p2buf = p1buf + (size_t)D * pstage;          // [D][T * AW]: second child

  if (threadIdx.x == 0) {
    sh.epoch = read_epoch(a.wait.sync);
    sh.abort = 0;
    for (int b = 0; b < D; ++b) {
      c_mbar_init(&sh.fullx[b], 1);
      c_mbar_init(&sh.fullp[b], 1);
      c_mbar_init(&sh.empty[b], kTreeConsumers);
    }
    for (int w = 0; w < kTreeConsumers; ++w) sh.done[w] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint32_t epoch = sh.epoch;
  const uint64_t E = (uint64_t)epoch << 32;
  const uint32_t tag = epoch + 1u;
  volatile uint32_t* abort = &sh.abort;

  // the two parts of the message, in units
  const size_t units = (a.count + PU - 1) / PU, whole = a.count / PU;
  const size_t ulo[2] = {0, a.half_units}, uhi[2] = {a.half_units, units};
  const size_t per_iter_units = (size_t)C * G * T;
  TreeSeq seq;
  uint32_t Q = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const TreeRole& R = t == 0 ? R0 : R1;
    const uint32_t iters = (uint32_t)((uhi[t] - ulo[t] + per_iter_units - 1) / per_iter_units);
    seq.lo[t] = 0;
    seq.hi[t] = R.leaf ? 0u : iters;
    seq.lo[2 + t] = L;
    seq.hi[2 + t] = R.root ? L : L + iters;
    Q += (seq.hi[t] - seq.lo[t] + seq.hi[2 + t] - seq.lo[2 + t]) * (uint32_t)G;
  }
  seq.tend = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) seq.tend = seq.hi[c] > seq.tend ? seq.hi[c] : seq.tend;
  auto tile_of = [&](const TreeCursor& k, uint32_t* nu, uint32_t* nx) -> size_t {
    const int t = k.tree();
    const size_t hi = t ? uhi[1] : uhi[0];
    const size_t base = (t ? ulo[1] : ulo[0]) + (((size_t)k.tile_it(L) * C + ch) * G + k.g) * (size_t)T;
    *nu = base < hi ? (uint32_t)(hi - base < (size_t)T ? hi - base : (size_t)T) : 0u;
    *nx = base < whole ? (uint32_t)(whole - base < (size_t)*nu ? whole - base : (size_t)*nu) : 0u;
    return base;
  };

  // links of this CTA (per channel): up FIFO slots, heads, up tails
  const size_t link_stride = (size_t)K * a.slot_bytes;
  auto up_fifo = [&](int node) { return a.fifo + ((size_t)node * C + ch) * link_stride; };
  auto up_head = [&](int node) { return a.head + (size_t)node * C + ch; };
  auto dn_head = [&](int node) { return a.head + (size_t)(n + node) * C + ch; };
  auto up_tail = [&](int node) { return a.tail + (size_t)node * C + ch; };
  const bool active = r != a.wait.skip_rank;
  // joined flags: each CTA marks its (rank, channel) for this call before
  // any wait, so an expired wait can tell a rank that never took part from
  // one stuck behind it (a tree's inner ranks post nothing until their
  // subtree has)
  auto joined = [&](int node) { return a.joined + (size_t)node * C + ch; };
  if (active && threadIdx.x == 0) st_relaxed(joined(r), E | 1u);

  if (active && warp <= kTreePLoaders) {
    // ---------------- loaders: warp 0 the own input, warps 1..P the incoming slots ----------------
    const bool px = warp == 0;
    const uint32_t np = (uint32_t)min(kTreePLoaders, D);
    const uint32_t mine = px ? 0u : (uint32_t)(warp - 1);
    uint32_t pos = 0;
    uint64_t* full = px ? sh.fullx : sh.fullp;
    TreeCursor k(seq);
    StagedStage st;
    uint32_t up_in = 0, up_out = 0, dn_in0 = 0, dn_in1 = 0;  // down messages received per tree
    // last value seen of each polled counter: the children's up heads, or
    // a leaf child's joined flag (0, 1), the up link's tail (2), the
    // parents' down heads in tree 0 and tree 1 (3, 4) -- one cache per
    // counter, never shared
    uint64_t seen[5] = {0, 0, 0, 0, 0};
    uint32_t q = 0;
    if (mine >= np) q = Q;
    for (; q < Q; ++q, k.next(G, seq), st.next(D), pos = pos + 1 == np ? 0u : pos + 1) {
      const bool up = k.up();
      const int tr = k.tree();
      uint32_t nu, nx;
      const size_t base = tile_of(k, &nu, &nx);
      const bool send_up = up && !Rp.root;
      if (!px && pos != mine) {  // another P loader's message: only count it
        if (up) {
          ++up_in;
          if (send_up) ++up_out;
        } else {
          ++(tr ? dn_in1 : dn_in0);
        }
        continue;
      }
      int ok = 1;
      if (lane == 0 && q >= (uint32_t)D && !staged_mbar_wait(&sh.empty[st.b], st.ph ^ 1u, abort, a.wait.timeout_ns)) {
        if (!*abort) record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, (int)q, tag);
        ok = 0;
      }
      const int parent = tr ? R1.parent : R0.parent;
      if (!px && ok) {
        // lanes 0/1: incoming heads (children, or the parent); lane 2: the
        // up link's tail; side by side
        const uint64_t* f = nullptr;
        uint64_t want = 0;
        int peer = -1, slot = 0;
        if (up && lane < Rp.nk) {
          // an inner child posts its partial; a leaf child only has to have
          // joined the call before its input is read
          const bool leaf_kid = lane == 0 ? Rp.lc[0] : Rp.lc[1];
          peer = lane == 0 ? Rp.kid[0] : Rp.kid[1];
          f = leaf_kid ? joined(peer) : up_head(peer);
          want = E | (uint64_t)(leaf_kid ? 1u : up_in + 1);
          slot = lane;
        } else if (!up && lane == 0) {
          f = dn_head(parent);
          want = E | (uint64_t)((tr ? dn_in1 : dn_in0) + 1);
          peer = parent;
          slot = 3 + tr;
        } else if (lane == 2 && send_up && up_out >= (uint32_t)K) {
          f = up_tail(r);
          want = E | (uint64_t)(up_out - K + 1);
          peer = Rp.parent;
          slot = 2;
        }
        if (f && seen[slot] < want) ok = wait_geq(f, want, &seen[slot], a.wait, tag, r, peer, (int)q, joined(peer));
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        if (px) {
          const uint32_t bytes = up ? nx * 16u : 0u;
          c_mbar_arrive_tx(&full[st.b], bytes);
          if (bytes)
            bulk_load_stream(xbuf + (size_t)st.b * xstage, static_cast<const char*>(a.in[r]) + base * 16, bytes,
                             &full[st.b]);
        } else {
          // partials: every unit of the tile from an inner child's slot, the
          // whole units of a leaf child's input; the total: the whole units
          // from the parent's output
          uint32_t each[2] = {0u, 0u};
          if (up) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
              if (i < Rp.nk) each[i] = Rp.lc[i] ? nx * 16u : nu * 16u * (uint32_t)AW;
          } else {
            each[0] = nx * 16u;
          }
          const uint32_t bytes = each[0] + each[1];
          if (bytes) fence_proxy_async_global();
          c_mbar_arrive_tx(&full[st.b], bytes);
          if (bytes) {
            if (up) {
              const size_t so = (size_t)(up_in % (uint32_t)K) * a.slot_bytes;
              unsigned char* dst[2] = {p1buf + (size_t)st.b * pstage, p2buf + (size_t)st.b * pstage};
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const int c = Rp.kid[i];
                if (i >= Rp.nk || each[i] == 0u) continue;
                if (Rp.lc[i])
                  bulk_load_stream(dst[i], static_cast<const char*>(a.in[c]) + base * 16, each[i], &full[st.b]);
                else
                  c_bulk_load(dst[i], up_fifo(c) + so, each[i], &full[st.b]);
              }
            } else {
              c_bulk_load(p1buf + (size_t)st.b * pstage, static_cast<const char*>(a.out[parent]) + base * 16,
                          each[0], &full[st.b]);
            }
          }
        }
      }
      if (up) {
        ++up_in;
        if (send_up) ++up_out;
      } else {
        ++(tr ? dn_in1 : dn_in0);
      }
    }
    if (q < Q && lane == 0) {
      *abort = 1;
      StagedStage w;
      const uint32_t lo = q > (uint32_t)D ? q - D : 0;
      for (uint32_t j = 0; j < q; ++j, w.next(D))
        if (j >= lo && (px || j % np == mine)) c_mbar_wait(&full[w.b], w.ph, a.wait.timeout_ns);
    }
  } else if (active && warp == kTreeSignaller) {
    // ---------------- signaller ----------------
    TreeCursor k(seq);
    uint32_t q = 0, up_out = 0, dn_out = 0;
    uint64_t t0 = 0;
    uint32_t spins = 0;
    while (q < Q) {
      uint32_t d = 0xffffffffu;
      if (lane < kTreeConsumers) d = ld_acquire_cta_u32(&sh.done[lane]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d = min(d, __shfl_xor_sync(0xffffffffu, d, o));
      if (d > q) {
        uint32_t nup = 0, ndn = 0;
        for (; q < d; ++q, k.next(G, seq)) {
          if (k.up()) {
            if (!Rp.root) ++nup;
            else if (Rp.nk > 0) ++ndn;  // a root posts its totals
          } else if ((k.tree() ? R1.nk : R0.nk) > 0) {
            ++ndn;
          }
        }
        if ((nup || ndn) && lane == 0) {
          fence_acq_rel();
          if (nup) red_max_relaxed(up_head(r), E | (uint64_t)(up_out + nup));
          if (ndn) red_max_relaxed(dn_head(r), E | (uint64_t)(dn_out + ndn));
        }
        up_out += nup;
        dn_out += ndn;
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
      __nanosleep(spins < 8 ? 32 : 128);
    }
  } else if (active && warp >= kTreeFirstConsumer) {
    // ---------------- consumers ----------------
    const int cw = warp - kTreeFirstConsumer;
    const int tid = cw * 32 + lane;
    TreeCursor k(seq);
    StagedStage st;
    uint32_t up_in = 0, up_slot = 0;
    const char* xg = static_cast<const char*>(a.in[r]);
    char* yg = static_cast<char*>(a.out[r]);
    for (uint32_t q = 0; q < Q; ++q, k.next(G, seq), st.next(D)) {
      const bool up = k.up();
      const int tr = k.tree();
      uint32_t nu, nx;
      const size_t base = tile_of(k, &nu, &nx);
      const bool send_up = up && !Rp.root;
      // a node with children keeps the total it stores in L2 for them
      const bool send_dn = up ? (Rp.root && Rp.nk > 0) : (tr ? R1.nk : R0.nk) > 0;
      const char* pg = static_cast<const char*>(a.out[tr ? R1.parent : R0.parent]);
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
      mbar_try_cta(&sh.fullx[st.b], st.ph);
      mbar_try_cta(&sh.fullp[st.b], st.ph);
      // the inner children's slots copied out: credits
      if (tid == 0 && up) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (i < Rp.nk && !Rp.lc[i]) red_max_relaxed(up_tail(Rp.kid[i]), E | (uint64_t)(up_in + 1));
      }
      const unsigned char* xs = xbuf + (size_t)st.b * xstage;
      const unsigned char* p1 = p1buf + (size_t)st.b * pstage;
      const unsigned char* p2 = p2buf + (size_t)st.b * pstage;
      char* so = send_up ? up_fifo(r) + (size_t)up_slot * a.slot_bytes : nullptr;
      for (uint32_t u = tid; u < nu; u += kTreeNT) {
        const size_t gu = base + u;
        const int v = unit_valid<DT>(gu, a.count);
        if (!up) {
          // the total, in the element type, from the parent's output; kept
          // in L2 when the children will read it
          const uint4 val = u < nx ? lds128(p1 + (size_t)u * 16) : ld_partial_l2<DT>(pg + gu * 16, v);
          if (send_dn)
            store_out<DT, true, false>(yg, gu, v, val);
          else
            store_out<DT, true, true>(yg, gu, v, val);
          continue;
        }
        Acc s;
        acc_init<DT>(s, u < nx ? lds128(xs + (size_t)u * 16) : ld_partial<DT>(xg + gu * 16, v));
        // the first child's partial, then the second's: accumulator words
        // from an inner child, the element type from a leaf's input
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i >= Rp.nk) break;
          const unsigned char* pi = i == 0 ? p1 : p2;
          if (Rp.lc[i]) {
            const char* cg = static_cast<const char*>(a.in[Rp.kid[i]]);
            acc_add<DT>(s, u < nx ? lds128(pi + (size_t)u * 16) : ld_partial<DT>(cg + gu * 16, v));
          } else {
            uint4 w[2];
#pragma unroll
            for (int qq = 0; qq < AW; ++qq) w[qq] = lds128(pi + ((size_t)u * AW + qq) * 16);
            acc_add_words<DT>(s, w);
          }
        }
        if (send_up) {
          uint4 o[2];
          acc_to_words<DT>(s, o);
#pragma unroll
          for (int qq = 0; qq < AW; ++qq) st_l2(so + ((size_t)u * AW + qq) * 16, o[qq]);
        } else {
          // root: the total, rounded once
          const uint4 val = acc_narrow<DT>(s);
          if (send_dn)
            store_out<DT, true, false>(yg, gu, v, val);
          else
            store_out<DT, true, true>(yg, gu, v, val);
        }
      }
      __syncwarp();
      if (lane == 0) {
        c_mbar_arrive_tx(&sh.empty[st.b], 0);
        st_release_cta_u32(&sh.done[cw], q + 1);
      }
      if (up) {
        ++up_in;
        if (send_up && ++up_slot == (uint32_t)K) up_slot = 0;
      }
    }
  }
  arrive_end(a.wait.sync, epoch);
}

template <int DT>
static const void* tree_staged_fn() {
  return reinterpret_cast<const void*>(&tree_staged_kernel<DT>);
}

static const void* tree_staged_pick(int dt) {
  if (dt == RRA_INT32) return tree_staged_fn<RRA_INT32>();
  if (dt == RRA_FLOAT32) return tree_staged_fn<RRA_FLOAT32>();
  if (dt == RRA_BFLOAT16) return tree_staged_fn<RRA_BFLOAT16>();
  return nullptr;
}

size_t tree_staged_smem(int dt, int tile_units, int stages) {
  const size_t aw = dt == RRA_BFLOAT16 ? 2 : 1;
  return (size_t)stages * (size_t)tile_units * 16 * (1 + 2 * aw);
}

cudaError_t tree_staged_occupancy(int dt, int tile_units, int stages, int* max_blocks_per_sm) {
  const void* f = tree_staged_pick(dt);
  if (!f || stages < 1 || stages > kTreeMaxStages) return cudaErrorInvalidValue;
  const size_t smem = tree_staged_smem(dt, tile_units, stages);
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, f, kTreeThreads, smem);
}

cudaError_t launch_tree_staged(int dt, const StagedTreeArgs& a, int grid, cudaStream_t s) {
  const void* f = tree_staged_pick(dt);
  if (!f || a.stages < 1 || a.stages > kTreeMaxStages) return cudaErrorInvalidValue;
  const size_t smem = tree_staged_smem(dt, a.slice_units, a.stages);
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<StagedTreeArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace rra
