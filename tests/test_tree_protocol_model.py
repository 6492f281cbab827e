"""A discrete-event model of the staged tree's link protocol
(kernels_tree_staged.cu), run on the CPU under random interleavings.

Nodes are virtual ranks in heap order (parent of r is (r-1)/2).  A leaf's
partial is its own input: it sends nothing up, and its parent reads the
tile from the leaf's input.  Each inner non-root node r owns an up FIFO
(its partial sums, read by its parent) of K
slots with a head counter (messages posted by the writer's signaller) and a
tail counter (messages the parent has copied out); the writer may reuse a
slot once the tail has passed it.  The totals come down without a FIFO: a
node with children stores each total in its own output and posts it on its
down head counter, and both children read it from there (an output is
written once, so it needs no credit).  A node's message
sequence is, per iteration of G tiles: its G up messages, then (not at the
root) the G down messages of the previous iteration, so the down wave of
one iteration overlaps the up wave of the next.  Per CTA the roles are as
in the staged ring: an X loader, P loaders taking messages round-robin (at
most as many as stages), in-order consumers, a signaller; stages are
tested by mbarrier phase parity.

Checked: every run finishes (no deadlock), no slot is read before it is
written or after it is reused, no output is read before it is posted, no
parity test passes for a phase that has not completed, and every rank ends
with the total summed in the order of
"Collective communication: NCCL's algorithms and protocols ...", section
"Algorithms" (tree), as the oracle reads it: p_r = (x_r + p_{2r+1}) + p_{2r+2}.
"""
import random

import pytest


class Aliasing(Exception):
    pass


def is_leaf(n, r):
    return r > 0 and 2 * r + 1 >= n


def tree_messages(n, r, G, iters, lag=1):
    if is_leaf(n, r):  # sends nothing up: only the totals coming down
        return [("dn", it, g) for it in range(iters) for g in range(G)]
    seq = []
    for it in range(iters + lag):
        if it < iters:
            for g in range(G):
                seq.append(("up", it, g))
        if it >= lag and r > 0:
            for g in range(G):
                seq.append(("dn", it - lag, g))
    return seq


def cursor_sequence(n, r, G, iters, lag):
    """The kernel's message cursor (TreeCursor) restated: after the up
    messages of iteration it come the down messages of iteration it - lag;
    once the ups are done, the remaining downs."""
    root, leaf = r == 0, is_leaf(n, r)
    Q = iters * G * (1 if root or leaf else 2)
    it, ph, g = (lag, 1, 0) if leaf else (0, 0, 0)
    seq = []
    for _ in range(Q):
        seq.append(("up", it, g) if ph == 0 else ("dn", it - lag, g))
        g += 1
        if g < G:
            continue
        g = 0
        if leaf:
            it += 1
            continue
        if ph == 0 and not root and it >= lag:
            ph = 1
            continue
        it += 1
        if it >= iters:
            it = max(it, lag)
            ph = 1
        else:
            ph = 0
    return seq


def children(n, r):
    return [c for c in (2 * r + 1, 2 * r + 2) if c < n]


def run_model(n, G, K, D, P, iters, seed, lag=1):
    rnd = random.Random(seed)
    seqs = [tree_messages(n, r, G, iters, lag) for r in range(n)]
    npl = min(P, D)
    # per rank: ordinals of up / down messages received and sent
    info = []
    for r in range(n):
        kids = children(n, r)
        rows = []
        up_in = up_out = dn_in = dn_out = 0
        for kind, it, g in seqs[r]:
            m = {"kind": kind, "it": it, "g": g}
            if kind == "up":
                m["up_in"] = up_in if kids else None  # same ordinal for both children
                up_in += 1 if kids else 0
                if r > 0:
                    m["up_out"] = up_out
                    up_out += 1
                elif kids:
                    m["dn_out"] = dn_out
                    dn_out += 1
            else:
                m["dn_in"] = dn_in
                dn_in += 1
                if kids:
                    m["dn_out"] = dn_out
                    dn_out += 1
            rows.append(m)
        info.append(rows)
    Q = [len(s) for s in seqs]
    X = [0] * n
    Pq = [list(range(npl)) for _ in range(n)]
    C = [0] * n
    S = [0] * n
    up_head = [0] * n  # published by the writer's signaller
    dn_head = [0] * n
    up_tail = [0] * n  # raised by the parent
    up_pub = [0] * n
    dn_pub = [0] * n
    up_slots = [[None] * K for _ in range(n)]
    stage = [[None] * D for _ in range(n)]
    fullx = [[0] * D for _ in range(n)]
    fullp = [[0] * D for _ in range(n)]
    empty = [[0] * D for _ in range(n)]
    out = [dict() for _ in range(n)]

    def empty_passes(r, q):
        if q < D:
            return True
        bb, ph = q % D, (q // D) & 1
        passes = (empty[r][bb] & 1) != (ph ^ 1)
        if passes and empty[r][bb] < q // D:
            raise Aliasing(("empty", r, q))
        return passes

    def credit_ok(r, m):
        return not ("up_out" in m and m["up_out"] >= K and up_tail[r] < m["up_out"] - K + 1)

    def data_ok(r, m):
        if m["kind"] == "up":
            if m["up_in"] is None:
                return True
            return all(up_head[c] >= m["up_in"] + 1 for c in children(n, r) if not is_leaf(n, c))
        return dn_head[(r - 1) // 2] >= m["dn_in"] + 1

    while True:
        acts = []
        for r in range(n):
            q = X[r]
            if q < Q[r] and empty_passes(r, q):
                acts.append(("X", r, None))
            for p in range(npl):
                q = Pq[r][p]
                if q < Q[r] and empty_passes(r, q) and data_ok(r, info[r][q]) and credit_ok(r, info[r][q]):
                    acts.append(("P", r, p))
            q = C[r]
            if q < Q[r]:
                bb, ph = q % D, (q // D) & 1
                if (fullx[r][bb] & 1) != ph and (fullp[r][bb] & 1) != ph:
                    if fullx[r][bb] != q // D + 1 or fullp[r][bb] != q // D + 1:
                        raise Aliasing(("full", r, q))
                    acts.append(("C", r, None))
            if S[r] < C[r]:
                acts.append(("S", r, None))
        if not acts:
            break
        kind, r, p = rnd.choice(acts)
        if kind == "X":
            fullx[r][X[r] % D] += 1
            X[r] += 1
        elif kind == "P":
            q = Pq[r][p]
            m = info[r][q]
            if m["kind"] == "up" and m["up_in"] is not None:
                got = []
                for c in children(n, r):
                    if is_leaf(n, c):  # the leaf's input tile, there from the start
                        got.append(((m["it"], m["g"]), ("x%d" % c,)))
                        continue
                    sl = up_slots[c][m["up_in"] % K]
                    assert sl is not None and sl[0] == m["up_in"], ("up slot", r, q, c, sl)
                    got.append(sl[1])
                stage[r][q % D] = got
            elif m["kind"] == "dn":  # the parent's output, once posted
                par = (r - 1) // 2
                key = (m["it"], m["g"])
                assert key in out[par], ("output read before it was posted", r, q)
                stage[r][q % D] = [(key, out[par][key])]
            else:
                stage[r][q % D] = []
            fullp[r][q % D] += 1
            Pq[r][p] += npl
        elif kind == "C":
            q = C[r]
            m = info[r][q]
            key = (m["it"], m["g"])
            got = stage[r][q % D]
            kids = children(n, r)
            if m["kind"] == "up":
                for k_, c in enumerate(kids):  # credits to the inner children
                    if not is_leaf(n, c):
                        up_tail[c] = max(up_tail[c], m["up_in"] + 1)
                for v in got:
                    assert v[0] == key, ("wrong up message", v, key)
                val = ("x%d" % r,) + tuple(v[1] for v in got)  # own, then left, then right
                if r > 0:
                    up_slots[r][m["up_out"] % K] = (m["up_out"], (key, val))
                else:
                    out[r][key] = val
            else:
                v = got[0]
                assert v[0] == key, ("wrong down message", v, key)
                out[r][key] = v[1]
            empty[r][q % D] += 1
            C[r] += 1
        else:
            d = C[r]
            for j in range(S[r], d):
                m = info[r][j]
                if "up_out" in m:
                    up_pub[r] += 1
                if "dn_out" in m:
                    dn_pub[r] += 1
            up_head[r], dn_head[r] = up_pub[r], dn_pub[r]
            S[r] = d
    assert all(C[r] == Q[r] and S[r] == Q[r] for r in range(n)), ("deadlock", n, G, K, D, P)

    def nested(r):
        return ("x%d" % r,) + tuple(nested(c) for c in children(n, r))

    want = nested(0)
    for r in range(n):
        assert len(out[r]) == iters * G, (r, len(out[r]))
        for key, v in out[r].items():
            assert v == want, (r, key, v, want)


CASES = [(n, G, K, D, P) for n in (1, 2, 3, 5, 8) for G, K in ((1, 2), (2, 3), (4, 8)) for D, P in ((1, 4), (2, 2), (3, 4))]


@pytest.mark.parametrize("n,G,K,D,P", CASES)
def test_staged_tree_protocol(n, G, K, D, P):
    for seed in range(3):
        run_model(n, G, K, D, P, iters=3, seed=seed)


@pytest.mark.parametrize("lag", [2, 3, 5])
@pytest.mark.parametrize("n,G,K,D,P", [(n, G, G + 1, D, P) for n in (2, 3, 5, 8) for G in (1, 2, 4)
                                       for D, P in ((1, 4), (2, 2), (3, 4))])
def test_staged_tree_protocol_lag(n, G, K, D, P, lag):
    # the broadcast trailing the reduction by several iterations: still no
    # deadlock with K = G + 1, including fewer iterations than the lag
    for iters in (1, 2, 4, 7):
        run_model(n, G, K, D, P, iters=iters, seed=iters, lag=lag)


@pytest.mark.parametrize("lag", [1, 2, 3])
def test_cursor_matches_sequence(lag):
    for n in (1, 2, 5, 8):
        for r in range(n):
            for G in (1, 3):
                for iters in (1, 2, 3, 6):
                    assert cursor_sequence(n, r, G, iters, lag) == tree_messages(n, r, G, iters, lag)
