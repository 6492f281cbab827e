// tree.cuh -- the double binary tree's shape, shared by its two kernels
// (kernels_tree_staged.cu for large messages, kernels_tree_ll.cu for small
// ones).
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Algorithms": the tree is a
// double binary tree.  Tree 0 is the binary tree in heap order over the
// ranks (rank r at position r; position p has children 2p+1 and 2p+2),
// tree 1 the same tree over the ranks reversed (rank r at position
// n-1-r).  A node's partial is its own data, then its child 2p+1's partial,
// then its child 2p+2's: p = (x (+) p_{2p+1}) (+) p_{2p+2}.
#pragma once

#include "common.cuh"

namespace rra {

// rank at heap position `pos` of tree t
__device__ __forceinline__ int tree_rank_at(int t, int n, int pos) { return t == 0 ? pos : n - 1 - pos; }

// Rank r's place in tree t.
struct TreeRole {
  int parent;      // the parent's rank (the root: its own)
  int kid[2];      // the children's ranks, position 2p+1 first (-1: none)
  int nk;          // children
  bool root;       // position 0
  bool leaf;       // below the root, no children
  bool lc[2];      // child i is a leaf
};

__device__ __forceinline__ TreeRole tree_role(int t, int n, int r) {
  const int p = t == 0 ? r : n - 1 - r;
  TreeRole o;
  o.root = p == 0;
  o.parent = o.root ? r : tree_rank_at(t, n, (p - 1) / 2);
  o.nk = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = 2 * p + 1 + i;
    o.kid[i] = c < n ? tree_rank_at(t, n, c) : -1;
    o.lc[i] = c < n && 2 * c + 1 >= n;
    o.nk += c < n ? 1 : 0;
  }
  o.leaf = !o.root && o.nk == 0;
  return o;
}

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

}  // namespace rra
