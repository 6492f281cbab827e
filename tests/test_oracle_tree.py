"""Pins of the oracle's tree all-reduce (reduce up a binary tree in heap
order, broadcast down): brute force, the summation order by hand-derived
float32 values, and the per-rank traffic of the tree."""
import numpy as np
import pytest

import oracle
from collective_all_reduce_rank_gb300 import inputs

B25 = float(2 ** 25)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8])
def test_tree_int32_brute_force(n):
    xs = inputs.make_ranks(n, 1001, "int32", "bits", seed=n)
    s = np.zeros(1001, np.int64)
    for x in xs:
        s += x
    want = ((s + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32)
    outs, _, _ = oracle.allreduce("tree", xs, "int32")
    for o in outs:
        assert np.array_equal(o, want)


def test_tree_summation_order_pinned():
    """n = 4: node 1's child is 3, the root's children are 1 and 2, so the
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


@pytest.mark.parametrize("n", [2, 3, 4, 8])
def test_tree_traffic_and_bound(n):
    # each rank receives one partial per child and, unless it is the root,
    # the result once: children(r) * S + (r > 0) * S
    count = 4 * 64
    S = count * 4
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=n, sigma=1e-2)
    outs, sent, recv = oracle.allreduce("tree", xs, "float32")
    for r in range(n):
        kids = sum(1 for c in (2 * r + 1, 2 * r + 2) if c < n)
        assert recv[r] == kids * S + (S if r > 0 else 0)
        assert sent[r] == kids * S + (S if r > 0 else 0)
    x64 = np.stack([x.astype(np.float64) for x in xs])
    g = (n - 1) * 2.0 ** -24 / (1 - (n - 1) * 2.0 ** -24)
    assert np.all(np.abs(outs[0] - x64.sum(0)) <= g * np.abs(x64).sum(0))
    assert all(o.tobytes() == outs[0].tobytes() for o in outs)
