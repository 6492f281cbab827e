// kernels_tree_staged.cu -- tree all-reduce with whole-CTA messages staged in
// shared memory by bulk copies, links through L2 (the machinery of the
// staged ring, kernels_ring_staged.cu).
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Algorithms": tree -- reduce
// up the tree, then broadcast down it, in O(log n) steps.  The tree is one
// binary tree in heap order (parent of rank r is (r-1)/2, children 2r+1 and
// 2r+2); a node's partial is its own data, then its left child's partial,
// then its right child's: p_r = (x_r (+) p_{2r+1}) (+) p_{2r+2}.  The root
// rounds the total once and it travels down unchanged, so every rank holds
// the same bits.  bfloat16 partials travel as float32.
//
// One persistent cooperative launch of n x C CTAs; CTA (r, ch) is channel ch
// of rank r.  A leaf's partial is its own input, so a leaf sends nothing
// up: its parent bulk-copies the tile from the leaf's input once the leaf
// has joined the call (the leaf's "joined" flag), and the leaf only
// receives.  Per channel each inner non-root node owns an up FIFO (its
// partials, read by its parent) of K slots in the workspace, with a head
// counter (messages posted) and a tail counter (messages the parent has
// copied out).  The totals going down need no FIFO: a node with children
// stores the total in its own output, kept in L2, and posts it on its down
// head counter; both children bulk-copy it from there (an output is
// written once per call, so these reads need no credit).  A node's
// messages, per iteration of G tiles of T units: its G up messages, then
// -- not at the root -- the G down messages of iteration it - L, so the
// broadcast of one iteration overlaps the reduction of the next L.  Warp
// roles as in the staged ring: an X loader (bulk-copies the node's own
// input tile), P loaders (acquire the heads of the incoming links and the
// tail of the up link, then bulk-copy the children's slots or inputs or
// the parent's output; at most as many as stages, so the stage mbarriers'
// parity tests stay sound), consumers (add, write the up slot or the
// output), and a signaller (one fence per run of finished messages, then
// the head counters).  Every wait is bounded.
//
// Needs 16-byte aligned buffers.  The last tile's partial 16-byte unit is
// read and written element-wise by the consumers.
#include "staged.cuh"

namespace rra {

constexpr int kTreePLoaders = 3;
constexpr int kTreeConsumers = 8;
constexpr int kTreeSignaller = 1 + kTreePLoaders;
constexpr int kTreeFirstConsumer = kTreeSignaller + 1;
constexpr int kTreeThreads = (kTreeFirstConsumer + kTreeConsumers) * 32;
constexpr int kTreeMaxStages = 8;
constexpr int kTreeNT = kTreeConsumers * 32;

// Position in a node's message sequence: iteration `it`, phase (0 = up
// messages of tile iteration it, 1 = down messages of tile iteration
// it - L), slice g.  The down messages trail by L iterations; once the ups
// are done, the remaining downs follow.
struct TreeCursor {
  uint32_t it, ph, g = 0;
  bool leaf;
  // a leaf below the root sends nothing up (its parent reads its input):
  // it has only down messages, of tile iterations 0, 1, ...
  __device__ __forceinline__ TreeCursor(bool leaf_, uint32_t L)
      : it(leaf_ ? L : 0u), ph(leaf_ ? 1u : 0u), leaf(leaf_) {}
  __device__ __forceinline__ void next(int G, uint32_t iters, bool root, uint32_t L) {
    if (++g < (uint32_t)G) return;
    g = 0;
    if (leaf) {
      ++it;
      return;
    }
    if (ph == 0 && !root && it >= L) {
      ph = 1;  // the downs of iteration it - L
      return;
    }
    ++it;
    if (it >= iters) {
      if (it < L) it = L;
      ph = 1;
    } else {
      ph = 0;
    }
  }
  __device__ __forceinline__ uint32_t tile_it(uint32_t L) const { return ph == 0 ? it : it - L; }
};

struct TreeShared {
  uint64_t fullx[kTreeMaxStages];
  uint64_t fullp[kTreeMaxStages];
  uint64_t empty[kTreeMaxStages];
  uint32_t done[kTreeConsumers];
  uint32_t abort;
  uint32_t epoch;
};

// a += w, w in accumulator words (a partial sum from a child)
template <int DT>
__device__ __forceinline__ void acc_add_words(Acc& a, const uint4* w) {
  if constexpr (DT == RRA_INT32) {
    a.w[0] += w[0].x;
    a.w[1] += w[0].y;
    a.w[2] += w[0].z;
    a.w[3] += w[0].w;
  } else {
    constexpr int AW = Elem<DT>::kAccWords;
#pragma unroll
    for (int q = 0; q < AW; ++q) {
      const uint32_t v[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        a.w[4 * q + i] = __float_as_uint(__fadd_rn(__uint_as_float(a.w[4 * q + i]), __uint_as_float(v[i])));
    }
  }
}

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
  const bool root = r == 0;
  const int parent = root ? 0 : (r - 1) / 2;
  const int nk = (2 * r + 1 < n) + (2 * r + 2 < n);           // children
  const bool leaf = nk == 0 && !root;                         // sends nothing up
  // a child that is a leaf: its partial is its input, read from there
  const bool lc[2] = {2 * r + 1 < n && 4 * r + 3 >= n, 2 * r + 2 < n && 4 * r + 5 >= n};
  const size_t xstage = (size_t)T * 16, pstage = (size_t)T * 16 * AW;
  unsigned char* xbuf = smem;                                 // [D][T] units
  unsigned char* p1buf = smem + (size_t)D * xstage;           // [D][T * AW]: left child / parent
  unsigned char* p2buf = p1buf + (size_t)D * pstage;          // [D][T * AW]: right child

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

  const size_t units = (a.count + PU - 1) / PU, whole = a.count / PU;
  const size_t per_iter_units = (size_t)C * G * T;
  const uint32_t iters = (uint32_t)((units + per_iter_units - 1) / per_iter_units);
  const uint32_t Q = iters * (uint32_t)G * (root || leaf ? 1u : 2u);
  auto tile_of = [&](const TreeCursor& k, uint32_t* nu, uint32_t* nx) -> size_t {
    const size_t base = (((size_t)k.tile_it(L) * C + ch) * G + k.g) * (size_t)T;
    *nu = base < units ? (uint32_t)(units - base < (size_t)T ? units - base : (size_t)T) : 0u;
    *nx = base < whole ? (uint32_t)(whole - base < (size_t)T ? whole - base : (size_t)T) : 0u;
    return base;
  };

  // links of this CTA (per channel): up FIFO slots, heads, up tails
  const size_t link_stride = (size_t)K * a.slot_bytes;
  auto up_fifo = [&](int node) { return a.fifo + ((size_t)node * C + ch) * link_stride; };
  auto up_head = [&](int node) { return a.head + (size_t)node * C + ch; };
  auto dn_head = [&](int node) { return a.head + (size_t)(n + node) * C + ch; };
  auto up_tail = [&](int node) { return a.tail + (size_t)node * C + ch; };
  // the parent's output: the totals coming down
  const char* pg = static_cast<const char*>(a.out[parent]);
  const int c1 = 2 * r + 1, c2 = 2 * r + 2;
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
    TreeCursor k(leaf, L);
    StagedStage st;
    uint32_t up_in = 0, dn_in = 0, up_out = 0;
    // last value seen of each polled counter: the children's up heads, or
    // a leaf child's joined flag (0, 1), the up link's tail (2), the
    // parent's down head (3) -- one cache per counter, never shared
    uint64_t seen[4] = {0, 0, 0, 0};
    uint32_t q = 0;
    if (mine >= np) q = Q;
    for (; q < Q; ++q, k.next(G, iters, root, L), st.next(D), pos = pos + 1 == np ? 0u : pos + 1) {
      const bool up = k.ph == 0;
      uint32_t nu, nx;
      const size_t base = tile_of(k, &nu, &nx);
      const bool has_in = up ? nk > 0 : true;
      const bool send_up = up && !root;
      if (!px && pos != mine) {  // another P loader's message: only count it
        if (up) {
          if (nk > 0) ++up_in;
          if (send_up) ++up_out;
        } else {
          ++dn_in;
        }
        continue;
      }
      int ok = 1;
      if (lane == 0 && q >= (uint32_t)D && !staged_mbar_wait(&sh.empty[st.b], st.ph ^ 1u, abort, a.wait.timeout_ns)) {
        if (!*abort) record_error(a.wait.status, RRA_ERR_TIMEOUT, r, -1, (int)q, tag);
        ok = 0;
      }
      if (!px && ok) {
        // lanes 0/1: incoming heads (children, or the parent); lane 2: the
        // up link's tail; side by side
        const uint64_t* f = nullptr;
        uint64_t want = 0;
        int peer = -1, slot = 0;
        if (up && lane < nk) {
          // an inner child posts its partial; a leaf child only has to have
          // joined the call before its input is read
          peer = lane == 0 ? c1 : c2;
          f = lc[lane] ? joined(peer) : up_head(peer);
          want = E | (uint64_t)(lc[lane] ? 1u : up_in + 1);
          slot = lane;
        } else if (!up && lane == 0) {
          f = dn_head(parent);
          want = E | (uint64_t)(dn_in + 1);
          peer = parent;
          slot = 3;
        } else if (lane == 2 && send_up && up_out >= (uint32_t)K) {
          f = up_tail(r);
          want = E | (uint64_t)(up_out - K + 1);
          peer = parent;
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
            for (int i = 0; i < nk; ++i) each[i] = lc[i] ? nx * 16u : nu * 16u * (uint32_t)AW;
          } else {
            each[0] = nx * 16u;
          }
          const uint32_t bytes = has_in ? each[0] + each[1] : 0u;
          if (bytes) fence_proxy_async_global();
          c_mbar_arrive_tx(&full[st.b], bytes);
          if (bytes) {
            if (up) {
              const size_t so = (size_t)(up_in % (uint32_t)K) * a.slot_bytes;
              unsigned char* dst[2] = {p1buf + (size_t)st.b * pstage, p2buf + (size_t)st.b * pstage};
              for (int i = 0; i < nk; ++i) {
                const int c = i == 0 ? c1 : c2;
                if (each[i] == 0u) continue;
                if (lc[i])
                  bulk_load_stream(dst[i], static_cast<const char*>(a.in[c]) + base * 16, each[i], &full[st.b]);
                else
                  c_bulk_load(dst[i], up_fifo(c) + so, each[i], &full[st.b]);
              }
            } else {
              c_bulk_load(p1buf + (size_t)st.b * pstage, pg + base * 16, each[0], &full[st.b]);
            }
          }
        }
      }
      if (up) {
        if (nk > 0) ++up_in;
        if (send_up) ++up_out;
      } else {
        ++dn_in;
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
    TreeCursor k(leaf, L);
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
        for (; q < d; ++q, k.next(G, iters, root, L)) {
          const bool up = k.ph == 0;
          if (up && !root) ++nup;
          if (up ? (root && nk > 0) : nk > 0) ++ndn;
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
    TreeCursor k(leaf, L);
    StagedStage st;
    uint32_t up_in = 0, up_slot = 0;
    const char* xg = static_cast<const char*>(a.in[r]);
    char* yg = static_cast<char*>(a.out[r]);
    for (uint32_t q = 0; q < Q; ++q, k.next(G, iters, root, L), st.next(D)) {
      const bool up = k.ph == 0;
      uint32_t nu, nx;
      const size_t base = tile_of(k, &nu, &nx);
      const bool send_up = up && !root;
      const bool send_dn = up ? (root && nk > 0) : nk > 0;
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
        if (nk > 0 && !lc[0]) red_max_relaxed(up_tail(c1), E | (uint64_t)(up_in + 1));
        if (nk > 1 && !lc[1]) red_max_relaxed(up_tail(c2), E | (uint64_t)(up_in + 1));
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
        // the left child's partial, then the right child's: accumulator
        // words from an inner child, the element type from a leaf's input
        for (int i = 0; i < nk; ++i) {
          const unsigned char* pi = i == 0 ? p1 : p2;
          if (lc[i]) {
            const char* cg = static_cast<const char*>(a.in[i == 0 ? c1 : c2]);
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
        if (nk > 0) ++up_in;
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
