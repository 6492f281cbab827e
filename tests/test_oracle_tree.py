"""Pins of the oracle's tree all-reduce: the double binary tree of
"Collective communication: NCCL's algorithms and protocols, ...", section
"Algorithms" (reduce up, broadcast down, O(log n) steps), read as tree 0 =
the heap-order binary tree over the ranks, tree 1 = the same tree over the
ranks in reverse order, the first half of the message (chunk plan for two
parts) on tree 0 and the second on tree 1.  Pinned by brute force, by
summation orders derived by hand in float32, and by the per-rank traffic
the two trees imply."""
import numpy as np
import pytest

import oracle
from collective_all_reduce_rank_gb300 import inputs

B25 = float(2 ** 25)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("count", [1, 7, 1001])
def test_tree_int32_brute_force(n, count):
    xs = inputs.make_ranks(n, count, "int32", "bits", seed=n + count)
    s = np.zeros(count, np.int64)
    for x in xs:
        s += x
    want = ((s + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32)
    outs, _, _ = oracle.allreduce("tree", xs, "int32")
    for o in outs:
        assert np.array_equal(o, want)


def test_tree_summation_order_pinned_first_tree():
    """Two elements: the chunk plan for two parts puts both in the first
    part (a part is a whole 16-byte unit, 4 float32), so only tree 0 sums.
    n = 4: node 1's child is 3, the root's children are 1 and 2, so the
    total is (x0 + (x1 + x3)) + x2 in float32.  Column A: x = (0.5, 2^25,
    -2^25, 0): (0.5 + 2^25) - 2^25 = 0, while adding the children first,
    (2^25 - 2^25) + 0.5, would give 0.5.  Column B: x = (0.5, 2^25, 1,
    -2^25): (0.5 + (2^25 - 2^25)) + 1 = 1.5, while ascending order,
    ((0.5 + 2^25) + 1) - 2^25, gives 0 (2^25 + 1 rounds to 2^25)."""
    xs = [np.array(v, np.float32) for v in ([0.5, 0.5], [B25, B25], [-B25, 1.0], [0.0, -B25])]
    outs, _, _ = oracle.allreduce("tree", xs, "float32")
    for o in outs:
        assert o[0] == 0.0 and o[1] == 1.5
    asc, _, _ = oracle.allreduce("oneshot", xs, "float32")
    assert asc[0][1] == 0.0


def test_double_tree_summation_order_pinned():
    """n = 4, 8 float32 per rank, every element of rank r equal to x_r with
    x = (0.5, 2^25, 2, -2^25).  The chunk plan for two parts gives elements
    0..3 to tree 0 and 4..7 to tree 1.

    Tree 0 (rank r at heap position r): (x0 + (x1 + x3)) + x2
      = (0.5 + 0) + 2 = 2.5.
    Tree 1 (rank 3 - p at position p): the root is rank 3, its children are
      rank 2 (position 1) and rank 1 (position 2), and rank 2's child is
      rank 0 (position 3): (x3 + (x2 + x0)) + x1 = (-2^25 + 2.5) + 2^25.
      -2^25 + 2.5 = -33554429.5 lies where float32 steps by 2 and rounds to
      -33554430 = -2^25 + 2, so the total is 2.
    A single tree would give 2.5 everywhere; the halves swapped, 2 then 2.5;
    tree 1 built by shifting the ranks one place instead of reversing them
    (rank 1 at the root): (x1 + (x2 + x0)) + x3 = (2^25 + 2.5) - 2^25 = 4
    (float32 steps by 4 above 2^25); tree 1 adding its root's children first,
    (x3 + x1) + (x2 + x0) = 2.5; ascending order ((0.5 + 2^25) + 2) - 2^25
    = 0 (both additions round back to 2^25)."""
    x = [0.5, B25, 2.0, -B25]
    xs = [np.full(8, v, np.float32) for v in x]
    outs, _, _ = oracle.allreduce("tree", xs, "float32")
    want = np.array([2.5] * 4 + [2.0] * 4, np.float32)
    for o in outs:
        assert np.array_equal(o, want), o
    asc, _, _ = oracle.allreduce("oneshot", xs, "float32")
    assert np.all(asc[0] == 0.0)


def _heap_children(n, p):
    return [c for c in (2 * p + 1, 2 * p + 2) if c < n]


@pytest.mark.parametrize("n", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("count", [4 * 64, 4 * 64 + 3, 5])
def test_tree_traffic_and_bound(n, count):
    """Per tree and rank: one partial received per child and, below the
    root, the total once; the same bytes sent.  The halves come from the
    chunk plan for two parts (16-byte units)."""
    per = -(-count // 2)
    h = min(count, -(-per // 4) * 4)
    halves = [h * 4, (count - h) * 4]
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=n, sigma=1e-2)
    outs, sent, recv = oracle.allreduce("tree", xs, "float32")
    for r in range(n):
        want = 0
        for t, S in enumerate(halves):
            p = r if t == 0 else n - 1 - r
            want += (len(_heap_children(n, p)) + (p > 0)) * S
        assert recv[r] == want and sent[r] == want, (r, recv[r], sent[r], want)
    # every non-root node of each tree moves its part up once and down once
    assert sum(recv) == 2 * (n - 1) * count * 4
    x64 = np.stack([x.astype(np.float64) for x in xs])
    g = (n - 1) * 2.0 ** -24 / (1 - (n - 1) * 2.0 ** -24)
    assert np.all(np.abs(outs[0] - x64.sum(0)) <= g * np.abs(x64).sum(0))
    assert all(o.tobytes() == outs[0].tobytes() for o in outs)


@pytest.mark.parametrize("n", [2, 4, 6, 8])
def test_even_n_no_rank_is_inner_in_both_trees(n):
    """With n even the two trees complement each other: a rank that
    forwards partials in one tree is a leaf in the other, so no rank's
    traffic exceeds that of one inner node with two children on one half
    plus a leaf on the other, 3 * S/2 + S/2 = 2S (S the bytes per rank);
    a single heap-order tree puts 3S on its inner ranks."""
    count = 4 * 256
    S = count * 4
    xs = inputs.make_ranks(n, count, "int32", "int20", seed=n)
    _, sent, recv = oracle.allreduce("tree", xs, "int32")
    assert max(recv) <= 2 * S and max(sent) <= 2 * S
    # a leaf of one tree moves half the message there: every rank moves at
    # least S/2 up and down in each tree it is a leaf of
    assert min(recv) >= S


def test_tree_bf16_rounds_once():
    """bfloat16: the root rounds the float32 total once.  n = 3, 16
    elements (two 16-byte units: the first 8 on tree 0, the rest on tree 1).
    Tree 0's root is rank 0 (value 1) with children ranks 1 and 2 (2^-8
    each): (1 + 2^-8) + 2^-8 = 1 + 2^-7, exact in float32 and in bfloat16,
    whereas rounding to bfloat16 after each add would give 1 (1 + 2^-8 is a
    tie, rounded to the even 1).  Tree 1 sums (2^-8 + 2^-8) + 1, the same
    value."""
    one = 0x3F80
    eps = 0x3B80  # 2^-8
    a = np.array([one] * 16, np.uint16)
    b = np.array([eps] * 16, np.uint16)
    c = np.array([eps] * 16, np.uint16)
    outs, _, _ = oracle.allreduce("tree", [a, b, c], "bfloat16")
    want = oracle.f32_to_bf16(np.array([1.0 + 2.0 ** -7], np.float32))[0]
    for o in outs:
        assert np.all(o == want), o
