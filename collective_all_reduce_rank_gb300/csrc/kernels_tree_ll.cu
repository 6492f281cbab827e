// kernels_tree_ll.cu -- double binary tree all-reduce for small messages,
// LL lines on every edge.
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks": section "Algorithms" gives the tree
// (a double binary tree: reduce up, broadcast down, O(log n) steps) and
// section "Protocols" the LL lines (4 data bytes under a 4-byte flag,
// polled by the receiver, so no fence and no separate flag sit on a hop).
// The shape and the summation order are those of tree.cuh, the same as the
// staged tree's: the message is split in two by the chunk plan for two
// parts, units [0, half_units) reduced over tree 0 and the rest over tree 1;
// p = (x (+) p_{2p+1}) (+) p_{2p+2}; the root rounds its total once and the
// total travels down unchanged, so every rank holds the same bits.
//
// Design on one GPU: one persistent cooperative launch of n x C CTAs of 8
// warps.  A warp tile is 32 lanes x kTreeLLUnits units (one unit a lane);
// warp w of CTA (r, ch) takes tiles ch*8 + w, + 8C, ... of both parts, as
// does the same warp of every other rank, so each edge of a tile joins two
// warps that handle it in the same order.  Per tile:
//   up    acc = x; for each child, poll its up lines of the tile and add
//         them (accumulator words: bfloat16 partials travel as float32);
//         below the root, post acc as LL lines in the own up region; at the
//         root, round, store the output and post the total down;
//   down  below the root, poll the parent's down lines, store the output
//         and, with children, post the total in the own down region.
// A warp does every up of its tiles before any down, the tree where its
// rank is a leaf first (those ups wait for nothing), and its downs in the
// tree where it has children first.  Ups wait only on children's ups and
// downs only on parents' downs or the root's up, so no chain of waits
// closes on itself.  Every line is written once per call and carries the
// call's tag (bit 30 set, bit 31 clear: the LL ring's flags set bit 31), so
// a line left by an earlier call never matches.  Every poll is bounded.
#include "tree.cuh"

namespace rra {

// This call's LL flag: never 0, never equal to an LL ring flag.
__device__ __forceinline__ uint32_t tree_ll_flag(uint32_t tag) { return 0x40000000u | (tag & 0x3FFFFFFFu); }

template <int DT>
struct TreeLLWarp {
  static constexpr int PU = Elem<DT>::kPerUnit;
  static constexpr int AW = Elem<DT>::kAccWords;
  static constexpr int UPT = kTreeLLUnits;
  static constexpr int TU = 32 * UPT;  // units per warp tile

  const TreeLLArgs& a;
  int r, lane;
  uint32_t f, tag;
  uint64_t E;
  size_t units;

  __device__ __forceinline__ char* up_region(int node) const {
    return a.lines + (size_t)node * (a.up_bytes + a.dn_bytes);
  }
  __device__ __forceinline__ char* dn_region(int node) const { return up_region(node) + a.up_bytes; }

  // Poll the lines of this lane's valid units in `region` (NG 16-byte word
  // groups per unit, 32 bytes of lines each) until every line of the warp
  // carries the flag; w receives the data words.  False when the call gave
  // up (this wait expired, recorded against `peer`, or another did).
  template <int NG>
  __device__ __forceinline__ bool get(const char* region, size_t u0, const int* v, uint4 (*w)[NG], int peer,
                                      int index) const {
    bool done = false;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
      if (!done) {
        bool all = true;
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
          if (v[j] == 0) continue;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            unsigned long long l0, l1, l2, l3;
            const char* p = region + ((u0 + 32 * j) * NG + q) * 32;
            ld_ll_pair(p, l0, l1);
            ld_ll_pair(p + 16, l2, l3);
            all = all && (uint32_t)(l0 >> 32) == f && (uint32_t)(l1 >> 32) == f && (uint32_t)(l2 >> 32) == f &&
                  (uint32_t)(l3 >> 32) == f;
            w[j][q] = make_uint4((uint32_t)l0, (uint32_t)l1, (uint32_t)l2, (uint32_t)l3);
          }
        }
        done = all;
      }
      if (__all_sync(0xffffffffu, done)) return true;
      if (it == 0) t0 = globaltimer();
      int give_up = 0;
      if ((it & 15u) == 15u && lane == 0) {
        if (aborted(a.wait.status, tag)) {
          give_up = 1;
        } else if (globaltimer() - t0 > a.wait.timeout_ns || it >= kMaxSpin) {
          // the peer never started this call (its joined flag holds an
          // older epoch): the rank that failed, not one stuck behind it
          const bool root = (ld_acquire(a.joined + (size_t)peer * a.channels) >> 32) != (E >> 32);
          record_error(a.wait.status, RRA_ERR_TIMEOUT, r, peer, index, tag, root);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
      if (!done) __nanosleep(32);
    }
  }

  // Post NG word groups per valid unit as LL lines.
  template <int NG>
  __device__ __forceinline__ void put(char* region, size_t u0, const int* v, const uint4 (*w)[NG]) const {
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        char* p = region + ((u0 + 32 * j) * NG + q) * 32;
        st_ll_pair(p, f, w[j][q].x, w[j][q].y);
        st_ll_pair(p + 16, f, w[j][q].z, w[j][q].w);
      }
    }
  }

  // valid elements of this lane's units of the tile at `base` in part [.., hi)
  __device__ __forceinline__ void valid(size_t base, size_t hi, int* v) const {
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = base + 32 * j + lane;
      v[j] = u < hi ? unit_valid<DT>(u, a.count) : 0;
    }
  }

  // Up of the tile at `base` in tree t (part [.., hi)): the partial goes to
  // the parent, or, at the root, the total to the output and down.
  __device__ __forceinline__ bool up(const TreeRole& R, size_t base, size_t hi, int index) const {
    int v[UPT];
    valid(base, hi, v);
    const size_t u0 = base + lane;
    Acc s[UPT];
#pragma unroll
    for (int j = 0; j < UPT; ++j)
      if (v[j] > 0) acc_init<DT>(s[j], load_in<DT, true>(a.in[r], u0 + 32 * j, v[j]));
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (i >= R.nk) break;
      uint4 w[UPT][AW];
      if (!get<AW>(up_region(R.kid[i]), u0, v, w, R.kid[i], index)) return false;
#pragma unroll
      for (int j = 0; j < UPT; ++j)
        if (v[j] > 0) acc_add_words<DT>(s[j], w[j]);
    }
    if (!R.root) {
      uint4 w[UPT][AW];
#pragma unroll
      for (int j = 0; j < UPT; ++j)
        if (v[j] > 0) acc_to_words<DT>(s[j], w[j]);
      put<AW>(up_region(r), u0, v, w);
      return true;
    }
    uint4 t[UPT][1];
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      if (v[j] == 0) continue;
      t[j][0] = acc_narrow<DT>(s[j]);
      store_out<DT, true, true>(a.out[r], u0 + 32 * j, v[j], t[j][0]);
    }
    if (R.nk > 0) put<1>(dn_region(r), u0, v, t);
    return true;
  }

  // Down of the tile at `base` in tree t below the root.
  __device__ __forceinline__ bool down(const TreeRole& R, size_t base, size_t hi, int index) const {
    int v[UPT];
    valid(base, hi, v);
    const size_t u0 = base + lane;
    uint4 t[UPT][1];
    if (!get<1>(dn_region(R.parent), u0, v, t, R.parent, index)) return false;
#pragma unroll
    for (int j = 0; j < UPT; ++j)
      if (v[j] > 0) store_out<DT, true, true>(a.out[r], u0 + 32 * j, v[j], t[j][0]);
    if (R.nk > 0) put<1>(dn_region(r), u0, v, t);
    return true;
  }

  __device__ __forceinline__ void run(int gw, int GW) {
    const int n = a.n;
    const TreeRole R0 = tree_role(0, n, r), R1 = tree_role(1, n, r);
    // the tree where this rank has children (tree 1 when it has none)
    const int ti = R0.nk > 0 ? 0 : 1;
    // ups: the leaf's tree first (nothing to wait for), then the other
    for (int k = 0; k < 2; ++k) {
      const int t = k == 0 ? 1 - ti : ti;
      const TreeRole R = t ? R1 : R0;
      const size_t lo = t ? a.half_units : 0, hi = t ? units : a.half_units;
      int index = 0;
      for (size_t base = lo + (size_t)gw * TU; base < hi; base += (size_t)GW * TU, ++index)
        if (!up(R, base, hi, index)) return;
    }
    // downs: the tree where this rank forwards first
    for (int k = 0; k < 2; ++k) {
      const int t = k == 0 ? ti : 1 - ti;
      const TreeRole R = t ? R1 : R0;
      if (R.root) continue;
      const size_t lo = t ? a.half_units : 0, hi = t ? units : a.half_units;
      int index = 0;
      for (size_t base = lo + (size_t)gw * TU; base < hi; base += (size_t)GW * TU, ++index)
        if (!down(R, base, hi, index)) return;
    }
  }
};

template <int DT>
__global__ void __launch_bounds__(kTreeLLThreads) tree_ll_kernel(const __grid_constant__ TreeLLArgs a) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch;
  const int r = blockIdx.x % a.n, ch = blockIdx.x / a.n;
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5;
  if (r != a.wait.skip_rank) {
    const uint64_t E = (uint64_t)epoch << 32;
    if (threadIdx.x == 0) st_relaxed(a.joined + (size_t)r * a.channels + ch, E | 1u);
    TreeLLWarp<DT> w{a, r, (int)(threadIdx.x & 31), tree_ll_flag(epoch + 1u), epoch + 1u, E,
                     (a.count + Elem<DT>::kPerUnit - 1) / Elem<DT>::kPerUnit};
    w.run(ch * W + warp, a.channels * W);
  }
  arrive_end(a.wait.sync, epoch);
}

static const void* tree_ll_pick(int dt) {
  if (dt == RRA_INT32) return reinterpret_cast<const void*>(&tree_ll_kernel<RRA_INT32>);
  if (dt == RRA_FLOAT32) return reinterpret_cast<const void*>(&tree_ll_kernel<RRA_FLOAT32>);
  if (dt == RRA_BFLOAT16) return reinterpret_cast<const void*>(&tree_ll_kernel<RRA_BFLOAT16>);
  return nullptr;
}

cudaError_t tree_ll_occupancy(int dt, int* max_blocks_per_sm) {
  const void* f = tree_ll_pick(dt);
  if (!f) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, f, kTreeLLThreads, 0);
}

cudaError_t launch_tree_ll(int dt, const TreeLLArgs& a, int grid, cudaStream_t s) {
  const void* f = tree_ll_pick(dt);
  if (!f) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTreeLLThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<TreeLLArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace rra
