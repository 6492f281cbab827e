"""The message-size sweep's largest point (1 GiB per rank) for every rank
count and type it times, against the oracle on sampled windows.

Inputs follow the sweep's seeded recipe (inputs.cfg_sweep, the seed the
sweep uses).  The oracle cannot sum n GiB in a test's time, so it computes
windows of the result: every element's sum depends only on that element of
each rank and on the order the schedule fixes for it, which the chunk it
falls in decides (the ring's rotation), or the part (the tree's two trees).
So each window set keeps that membership: for the ring, one-shot and
two-shot, a window of m elements from the start, the middle and the end of
every one of the n chunks forms a problem of n chunks of m elements; for the
tree, windows from both parts form a two-part problem.  The GPU's elements
at those positions must equal the oracle's bit for bit (bfloat16 also within
1e-2 relative), on every rank.
"""
import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

AR = {"ring": rra.RRA_ALGO_RING, "oneshot": rra.RRA_ALGO_ONE_SHOT, "twoshot": rra.RRA_ALGO_TWO_SHOT,
      "tree": rra.RRA_ALGO_TREE}
S_MAX = max(inputs.SWEEP_SIZES)
CASES = [(n, "int32") for n in inputs.SWEEP_RANKS] + [(n, "bfloat16") for n in inputs.SWEEP_RANKS] + \
        [(8, "float32")]


@pytest.fixture(scope="module", autouse=True)
def _init():
    import torch

    torch.cuda.set_device(0)
    rra.rra_init(0)
    rra.rra_set_timeout_ns(2_000_000_000)
    yield
    torch.cuda.empty_cache()


def _parts(count, parts, dtype):
    """Element bounds of the chunk plan for `parts` parts (whole 16-byte
    vectors per part; the same rule as the schedules)."""
    b = oracle.chunk_plan(parts, count, dtype)
    return [(b[i], b[i + 1]) for i in range(parts)]


def _windows(bounds, m):
    """Start, middle and end windows of m elements inside every part."""
    sets = []
    for where in ("start", "mid", "end"):
        win = []
        for lo, hi in bounds:
            off = lo if where == "start" else (hi - m if where == "end" else lo + (hi - lo) // 2 // 16 * 16)
            win.append(off)
        sets.append(win)
    return sets


@pytest.mark.parametrize("n,dtype", CASES)
def test_sweep_top_size_matches_oracle_on_windows(n, dtype):
    import torch

    import gpu_util as g

    xs = inputs.cfg_sweep(n, S_MAX, dtype, seed=S_MAX + n)
    count = xs[0].size
    ins = [g.to_dev(x, dtype) for x in xs]
    outs = g.empty(n, count, dtype)
    m = 256  # elements per window: whole 16-byte vectors for every type
    for name, algo in AR.items():
        for o in outs:
            o.view(torch.int16 if dtype == "bfloat16" else torch.int32).fill_(-1)
        rra.rra_allreduce(ins, outs, count, g.CODE[dtype], rra.RRA_SUM, algo)
        st, info = rra.rra_query_status()
        assert st == 0, (name, info)
        bounds = _parts(count, 2 if name == "tree" else n, dtype)
        for win in _windows(bounds, m):
            sub = [np.concatenate([x[o:o + m] for o in win]) for x in xs]
            want, _, _ = oracle.allreduce(name, sub, dtype)
            idx = np.concatenate([np.arange(o, o + m) for o in win])
            t_idx = torch.from_numpy(idx).cuda()
            for r in range(n):
                got = g.to_host(outs[r][t_idx], dtype)
                if dtype == "bfloat16":
                    assert g.bf16_rel_ok(got, want[r]), (name, r)
                g.assert_bits_equal(got, want[r], "%s n=%d %s r=%d windows %s" % (name, n, dtype, r, win[:2]))
    del ins, outs
    torch.cuda.empty_cache()
