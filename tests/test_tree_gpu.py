"""Tree all-reduce on the GPU vs the oracle's tree, bit for bit."""
import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _init():
    import torch

    torch.cuda.set_device(0)
    rra.rra_init(0)
    rra.rra_set_timeout_ns(2_000_000_000)
    yield


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n", [2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("count", [1, 7, 4096, 100_003, 3_000_001])
def test_tree_matches_oracle(dtype, n, count):
    import gpu_util as g

    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + n)
    want, _, _ = oracle.allreduce("tree", xs, dtype)
    for inplace in (False, True):
        ins = [g.to_dev(x, dtype) for x in xs]
        outs = ins if inplace else g.empty(n, count, dtype)
        rra.rra_allreduce(ins, outs, count, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_TREE)
        st, info = rra.rra_query_status()
        assert st == 0, info
        for r in range(n):
            got = g.to_host(outs[r], dtype)
            if dtype == "bfloat16":
                assert g.bf16_rel_ok(got, want[r])
            g.assert_bits_equal(got, want[r], "tree n=%d r=%d inplace=%s" % (n, r, inplace))


@pytest.mark.parametrize("tile,G,K,stages", [(1024, 4, 8, 8), (128, 1, 2, 1), (256, 3, 4, 2), (512, 8, 9, 3),
                                             (2048, 2, 3, 8)])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,count", [(2, 3), (3, 100_003), (5, 70_001), (8, 8 * 1024 * 4 * 19 + 7), (8, 3_000_001)])
def test_staged_tree_shapes(tile, G, K, stages, dtype, n, count, monkeypatch):
    # the staged tree over message sizes, tiles per iteration, FIFO depths
    # and pipeline depths, down to one slot of credit beyond G and one stage:
    # the oracle's tree bits, twice in a row and in place
    import gpu_util as g

    for k, v in (("RRA_TREE_TILE", tile), ("RRA_TREE_G", G), ("RRA_TREE_K", K), ("RRA_TREE_STAGES", stages),
                 ("RRA_TREE_PROTO", "staged")):
        monkeypatch.setenv(k, str(v))
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + n + tile)
    want, _, _ = oracle.allreduce("tree", xs, dtype)
    for inplace in (False, True):
        ins = [g.to_dev(x, dtype) for x in xs]
        outs = ins if inplace else g.empty(n, count, dtype)
        rra.rra_allreduce(ins, outs, count, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_TREE)
        st, info = rra.rra_query_status()
        assert st == 0, info
        for r in range(n):
            g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "staged tree n=%d r=%d" % (n, r))


@pytest.mark.parametrize("lag", [2, 3, 9])
@pytest.mark.parametrize("tile,G,K,stages", [(256, 3, 4, 2), (1024, 4, 5, 8), (128, 1, 2, 1)])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("n,count", [(2, 3), (5, 70_001), (8, 8 * 1024 * 4 * 19 + 7), (8, 3_000_001)])
def test_staged_tree_lag(lag, tile, G, K, stages, dtype, n, count, monkeypatch):
    # the broadcast trailing the reduction by several iterations (more than
    # the call has, too): the oracle's tree bits
    import gpu_util as g

    for k, v in (("RRA_TREE_TILE", tile), ("RRA_TREE_G", G), ("RRA_TREE_K", K), ("RRA_TREE_STAGES", stages),
                 ("RRA_TREE_LAG", lag), ("RRA_TREE_PROTO", "staged")):
        monkeypatch.setenv(k, str(v))
    xs = inputs.make_ranks(n, count, dtype, "normal", seed=count + n + lag)
    want, _, _ = oracle.allreduce("tree", xs, dtype)
    ins = [g.to_dev(x, dtype) for x in xs]
    outs = g.empty(n, count, dtype)
    rra.rra_allreduce(ins, outs, count, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_TREE)
    st, info = rra.rra_query_status()
    assert st == 0, info
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "staged tree lag=%d n=%d r=%d" % (lag, n, r))


@pytest.mark.parametrize("form", ["staged", "ll"])
def test_tree_order_case_on_gpu(form, monkeypatch):
    # the hand-derived n = 4 double-tree case of the oracle's pins, x =
    # (0.5, 2^25, 2, -2^25) on every element of each rank: 2.5 on the part
    # tree 0 sums, (x0 + (x1 + x3)) + x2, and 2 on tree 1's part,
    # (x3 + (x2 + x0)) + x1; many tiles in each part, in both forms
    import gpu_util as g

    monkeypatch.setenv("RRA_TREE_PROTO", form)
    B = float(2 ** 25)
    count = 4 * 40_000
    xs = [np.full(count, v, np.float32) for v in (0.5, B, 2.0, -B)]
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = g.empty(4, count, "float32")
    rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TREE)
    assert rra.rra_query_status()[0] == 0
    for r in range(4):
        got = g.to_host(outs[r], "float32")
        assert np.all(got[: count // 2] == 2.5) and np.all(got[count // 2:] == 2.0), r


def test_tree_rejects_unaligned():
    import gpu_util as g

    xs = inputs.make_ranks(2, 1001, "float32", "normal")
    ins = [g.to_dev(np.concatenate([[0.0], x]).astype(np.float32), "float32")[1:] for x in xs]
    outs = g.empty(2, 1001, "float32")
    st = rra.rra_allreduce(ins, outs, 1001, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TREE, check=False)
    assert st == rra.RRA_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,count", [(2, 1), (2, 400_003), (3, 7), (4, 4096), (5, 100_003), (7, 65_537),
                                     (8, 5), (8, 20_480), (8, 240_007)])
def test_ll_tree_matches_oracle(dtype, n, count, monkeypatch):
    # the LL form forced over shapes: one unit, ragged tails, one tile per
    # warp and several (8 x 240,007 fp32 and 2 x 400,003 loop their warps),
    # in place and out of place, twice in a row (every line carries the
    # call's tag, so the first call's lines never satisfy the second's polls)
    import gpu_util as g

    monkeypatch.setenv("RRA_TREE_PROTO", "ll")
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + n + 17)
    want, _, _ = oracle.allreduce("tree", xs, dtype)
    for inplace in (False, True):
        for rep in range(2):
            ins = [g.to_dev(x, dtype) for x in xs]
            outs = ins if inplace else g.empty(n, count, dtype)
            rra.rra_allreduce(ins, outs, count, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_TREE)
            st, info = rra.rra_query_status()
            assert st == 0, info
            for r in range(n):
                got = g.to_host(outs[r], dtype)
                if dtype == "bfloat16":
                    assert g.bf16_rel_ok(got, want[r])
                g.assert_bits_equal(got, want[r], "LL tree n=%d r=%d inplace=%s rep=%d" % (n, r, inplace, rep))


def test_ll_tree_too_large_for_its_region(monkeypatch):
    # forced LL on a message whose lines do not fit the LL region: a
    # workspace error, no launch
    import gpu_util as g

    monkeypatch.setenv("RRA_TREE_PROTO", "ll")
    n, count = 8, 1 << 22
    ins = [g.to_dev(np.ones(count, np.float32), "float32") for _ in range(n)]
    outs = g.empty(n, count, "float32")
    st = rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TREE, check=False)
    assert st == rra.RRA_ERR_WORKSPACE
    monkeypatch.setenv("RRA_TREE_PROTO", "staged")
    rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TREE)
    assert rra.rra_query_status()[0] == 0
    assert np.all(g.to_host(outs[3], "float32") == 8.0)


@pytest.mark.parametrize("max_ctas", [1, 8, 19])
@pytest.mark.parametrize("form", ["staged", "ll"])
def test_tree_under_sm_budget(max_ctas, form, monkeypatch):
    # an SM budget leaves the tree one or a few channels per rank: its warps
    # (LL) or CTAs (staged) loop over many tiles; the oracle's bits
    import gpu_util as g

    monkeypatch.setenv("RRA_TREE_PROTO", form)
    n, count = 8, 100_003
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=max_ctas + 7)
    want, _, _ = oracle.allreduce("tree", xs, "float32")
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = g.empty(n, count, "float32")
    rra.rra_set_max_ctas(max_ctas)
    try:
        rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TREE)
        st, info = rra.rra_query_status()
    finally:
        rra.rra_set_max_ctas(0)
    assert st == 0, info
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], "float32"), want[r], "tree %s max_ctas=%d r=%d" % (form, max_ctas, r))
