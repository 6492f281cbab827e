"""A model of the LL double tree's schedule (kernels_tree_ll.cu), run on the
CPU under random interleavings.

Each rank's warps handle the same tiles in the same order: first the up
step of every tile in the tree where the rank is a leaf (it waits for
nothing), then the up steps in the tree where it has children (each waits
for its children's up lines of that tile), then the down steps below the
root, the tree where it forwards first (each waits for the parent's down
lines of that tile).  An up step posts the node's partial, or at the root
the total, which it also stores; a down step stores the total and, with
children, posts it down.  Every line is written once per call.

Checked: every run finishes (no wait cycle), no line is read before it is
written and none is written twice, and every rank ends with each part's
total summed in the order of "Collective communication: NCCL's algorithms
and protocols ...", section "Algorithms" (the double binary tree), as the
oracle reads it: at each node p = (x + p_{2p+1}) + p_{2p+2}.
"""
import random

import pytest


def rank_at(t, n, pos):
    return pos if t == 0 else n - 1 - pos


def role(t, n, r):
    p = r if t == 0 else n - 1 - r
    kids = [rank_at(t, n, c) for c in (2 * p + 1, 2 * p + 2) if c < n]
    return {"root": p == 0, "parent": r if p == 0 else rank_at(t, n, (p - 1) // 2), "kids": kids}


def warp_program(n, r, tiles):
    """The ops of one warp of rank r: (kind, tree, tile), in kernel order."""
    R = [role(0, n, r), role(1, n, r)]
    ti = 0 if R[0]["kids"] else 1
    ops = []
    for t in (1 - ti, ti):
        ops += [("up", t, k) for k in tiles[t]]
    for t in (ti, 1 - ti):
        if not R[t]["root"]:
            ops += [("down", t, k) for k in tiles[t]]
    return ops


def run_model(n, tiles_per_part, warps, seed):
    rng = random.Random(seed)
    # warp w takes tiles w, w + warps, ... of each part (the same on every rank)
    progs = {}
    for r in range(n):
        for w in range(warps):
            tiles = [list(range(w, tiles_per_part[t], warps)) for t in (0, 1)]
            progs[(r, w)] = warp_program(n, r, tiles)
    pc = {k: 0 for k in progs}
    up_lines, dn_lines, out = {}, {}, {}

    def ready(r, op):
        kind, t, k = op
        R = role(t, n, r)
        if kind == "up":
            return all((c, t, k) in up_lines for c in R["kids"])
        return (R["parent"], t, k) in dn_lines

    def step(r, op):
        kind, t, k = op
        R = role(t, n, r)
        if kind == "up":
            acc = "x%d" % r
            for c in R["kids"]:
                acc = "(%s+%s)" % (acc, up_lines[(c, t, k)])
            if R["root"]:
                assert (r, t, k) not in out and (r, t, k) not in dn_lines, "written twice"
                out[(r, t, k)] = acc
                if R["kids"]:
                    dn_lines[(r, t, k)] = acc
            else:
                assert (r, t, k) not in up_lines, "up line written twice"
                up_lines[(r, t, k)] = acc
        else:
            total = dn_lines[(R["parent"], t, k)]
            assert (r, t, k) not in out, "output written twice"
            out[(r, t, k)] = total
            if R["kids"]:
                assert (r, t, k) not in dn_lines, "down line written twice"
                dn_lines[(r, t, k)] = total

    while True:
        live = [k for k in progs if pc[k] < len(progs[k])]
        if not live:
            break
        runnable = [k for k in live if ready(k[0], progs[k][pc[k]])]
        assert runnable, "deadlock: %s" % [(k, progs[k][pc[k]]) for k in live]
        k = rng.choice(runnable)
        step(k[0], progs[k][pc[k]])
        pc[k] += 1
    return out


def expected(n, t):
    """The oracle's order for tree t: p = (x + p_{2p+1}) + p_{2p+2}."""
    def part(pos):
        acc = "x%d" % rank_at(t, n, pos)
        for c in (2 * pos + 1, 2 * pos + 2):
            if c < n:
                acc = "(%s+%s)" % (acc, part(c))
        return acc
    return part(0)


@pytest.mark.parametrize("n", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("tiles,warps", [((1, 0), 1), ((1, 1), 1), ((3, 2), 2), ((5, 5), 2), ((4, 1), 3)])
@pytest.mark.parametrize("seed", range(4))
def test_ll_tree_schedule(n, tiles, warps, seed):
    out = run_model(n, tiles, warps, seed)
    for t in (0, 1):
        want = expected(n, t)
        for k in range(tiles[t]):
            for r in range(n):
                assert out[(r, t, k)] == want, (r, t, k)


def test_model_catches_a_wrong_order():
    # a kernel that waited for its down steps before its leaf ups would
    # deadlock: the model must report it
    global warp_program
    saved = warp_program

    def bad_program(n, r, tiles):
        ops = saved(n, r, tiles)
        return [o for o in ops if o[0] == "down"] + [o for o in ops if o[0] == "up"]

    warp_program = bad_program
    try:
        with pytest.raises(AssertionError, match="deadlock"):
            run_model(4, (1, 1), 1, 0)
    finally:
        warp_program = saved
