"""Failure detection on the GPU without a fault: a virtual rank that posts
nothing makes its peers' bounded waits expire; the kernel returns, the status
word names the rank, and the next call works.  No trap, no hang."""
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
    yield
    rra.rra_debug_skip_rank(-1)
    rra.rra_set_timeout_ns(0)


@pytest.mark.parametrize("algo,proto", [(rra.RRA_ALGO_RING, "simple"), (rra.RRA_ALGO_RING, "ll"),
                                        (rra.RRA_ALGO_RING, "staged"), (rra.RRA_ALGO_TWO_SHOT, None),
                                        (rra.RRA_ALGO_TREE, "staged"), (rra.RRA_ALGO_TREE, "ll")])
@pytest.mark.parametrize("skip", [0, 3])
def test_crashed_rank_times_out_and_gpu_stays_usable(algo, proto, skip, monkeypatch):
    import gpu_util as g

    if proto:
        monkeypatch.setenv("RRA_TREE_PROTO" if algo == rra.RRA_ALGO_TREE else "RRA_RING_PROTO", proto)
    n, count = 4, 1 << 16 if proto == "ll" and algo == rra.RRA_ALGO_TREE else 1 << 20
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=1)
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = g.empty(n, count, "float32")
    rra.rra_set_timeout_ns(1_000_000)  # 1 ms
    rra.rra_debug_skip_rank(skip)
    try:
        rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, algo)
        st, info = rra.rra_query_status()
    finally:
        rra.rra_debug_skip_rank(-1)
        rra.rra_set_timeout_ns(2_000_000_000)
    assert st == rra.RRA_ERR_TIMEOUT
    assert info[0] == rra.RRA_ERR_TIMEOUT
    assert info[2] == skip, info  # the rank waited for is the silent one
    # recovery: the next call on the same workspace is correct
    rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, algo)
    st, info = rra.rra_query_status()
    assert st == 0, info
    name = {rra.RRA_ALGO_RING: "ring", rra.RRA_ALGO_TREE: "tree"}.get(algo, "twoshot")
    want, _, _ = oracle.allreduce(name, xs, "float32")
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], "float32"), want[r], "after recovery")


@pytest.mark.parametrize("skip", [0, 3])
def test_static_two_shot_silent_rank_times_out_and_recovers(skip):
    # the allocation-free two-shot honours the wait bound and the fault
    # injection, and reports through its own status query
    import gpu_util as g

    n, count = 4, 1 << 20
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=2)
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = g.empty(n, count, "float32")
    rra.rra_set_timeout_ns(1_000_000)  # 1 ms
    rra.rra_debug_skip_rank(skip)
    try:
        rra.rra_allreduce_two_shot_static(ins, outs, count, rra.RRA_FLOAT32)
        st, info = rra.rra_query_status_static()
    finally:
        rra.rra_debug_skip_rank(-1)
        rra.rra_set_timeout_ns(2_000_000_000)
    assert st == rra.RRA_ERR_TIMEOUT and info[0] == rra.RRA_ERR_TIMEOUT
    assert info[2] == skip, info
    # the status was read and cleared; the next call is correct
    rra.rra_allreduce_two_shot_static(ins, outs, count, rra.RRA_FLOAT32)
    st, info = rra.rra_query_status_static()
    assert st == 0, info
    want, _, _ = oracle.allreduce("twoshot", xs, "float32")
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], "float32"), want[r], "static after recovery")
    # the regular status word saw none of it
    assert rra.rra_query_status()[0] == 0


@pytest.mark.parametrize("skip", [0, 6])
def test_split_two_shot_silent_rank_times_out_and_recovers(skip):
    # the split two-shot (five ranks and more: reducer and gatherer warps):
    # the gatherers' bounded waits name the silent rank; the next call is
    # correct
    import gpu_util as g

    n, count = 8, (1 << 20) + 5
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=3)
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = g.empty(n, count, "float32")
    rra.rra_set_timeout_ns(1_000_000)  # 1 ms
    rra.rra_debug_skip_rank(skip)
    try:
        rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TWO_SHOT)
        st, info = rra.rra_query_status()
    finally:
        rra.rra_debug_skip_rank(-1)
        rra.rra_set_timeout_ns(2_000_000_000)
    assert st == rra.RRA_ERR_TIMEOUT and info[2] == skip, info
    rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TWO_SHOT)
    assert rra.rra_query_status()[0] == 0
    want, _, _ = oracle.allreduce("twoshot", xs, "float32")
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], "float32"), want[r], "split two-shot after recovery")


def test_flight_recorder_lists_recent_calls():
    import gpu_util as g

    xs = inputs.make_ranks(2, 1000, "int32", "int20")
    ins = [g.to_dev(x, "int32") for x in xs]
    outs = g.empty(2, 1000, "int32")
    rra.rra_allreduce(ins, outs, 1000, rra.RRA_INT32, rra.RRA_SUM, rra.RRA_ALGO_ONE_SHOT)
    rra.rra_allreduce(ins, outs, 1000, rra.RRA_INT32, rra.RRA_SUM, rra.RRA_ALGO_RING)
    text = rra.rra_dump_recent().strip().splitlines()
    assert "allreduce algo=one_shot n=2 count=1000 dtype=int32" in text[-2]
    assert "allreduce algo=ring n=2 count=1000 dtype=int32" in text[-1]
    assert text[-1].endswith("status=success")
