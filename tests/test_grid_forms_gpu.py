"""One-shot, direct reduce-scatter and direct all-gather on both sides of
the size at which their launch switches from a resident grid-stride grid to
a grid that covers the message (256 MB of floor bytes for one-shot, 64 MB
for the reduce-scatter and all-gather; every thread one trip of `upt`
units): the same sums bit for bit as the oracle on either side, aligned and
ragged, and the recorded grid is the covering one above the threshold only."""
import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = pytest.mark.gpu

ONESHOT_FROM = 256 << 20  # floor bytes from which one-shot covers
DIRECT_FROM = 64 << 20    # the same for the direct reduce-scatter and all-gather
ES = {"float32": 4, "bfloat16": 2}


@pytest.fixture(scope="module", autouse=True)
def _init():
    import torch

    torch.cuda.set_device(0)
    rra.rra_init(0)
    rra.rra_set_timeout_ns(2_000_000_000)
    yield


def G():
    import gpu_util

    return gpu_util


def _last_grid():
    line = rra.rra_dump_recent().strip().splitlines()[-1]
    assert "status=success" in line, line
    return int(line.split("grid=")[1].split()[0])


def _cover(units, upt):
    """The covering grid's CTAs (per row) for `units` units, 512 threads."""
    return -(-units // (512 * upt))


def _units_from(floor_from, floor_per_unit):
    """The fewest 16-byte units whose floor bytes reach the threshold."""
    return -(-floor_from // floor_per_unit)


def _count_for(units, e, ragged):
    """Element count with `units` 16-byte units (the last one partial when
    ragged)."""
    pu = 16 // e
    return units * pu - (pu - 1 if ragged else 0)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("n", [2, 4, 8])
def test_oneshot_either_side(dtype, n):
    g = G()
    e = ES[dtype]
    t = _units_from(ONESHOT_FROM, 2 * n * 16)
    upt = 2 if n <= (3 if dtype == "bfloat16" else 4) else 1  # units a thread takes in one trip
    grids = []
    for units, ragged in ((t - 1, False), (t + 1, True)):
        count = _count_for(units, e, ragged)
        xs = inputs.make_ranks(n, count, dtype, "normal", seed=units + n)
        ins = [g.to_dev(x, dtype) for x in xs]
        outs = g.empty(n, count, dtype)
        rra.rra_allreduce(ins, outs, count, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_ONE_SHOT)
        grids.append((_last_grid(), _cover(units, upt)))
        want, _, _ = oracle.allreduce("oneshot", xs, dtype)
        for r in (0, n - 1):
            g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "one-shot n=%d units=%d r=%d" % (n, units, r))
        del ins, outs
    (below, below_cover), (above, above_cover) = grids
    assert below != below_cover and above == above_cover, grids


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("n", [2, 8])
def test_direct_rs_ag_either_side(dtype, n):
    g = G()
    e = ES[dtype]
    t = _units_from(DIRECT_FROM, (n + 1) * n * 16)
    rs_grids, ag_grids = [], []
    for units, ragged in ((t - 1, False), (t + 1, True)):
        rc = _count_for(units, e, ragged)
        xs = inputs.make_ranks(n, n * rc, dtype, "normal", seed=units + 7 * n)
        ins = [g.to_dev(x, dtype) for x in xs]
        outs = g.empty(n, rc, dtype)
        rra.rra_reduce_scatter(ins, outs, rc, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_DIRECT)
        rs_grids.append((_last_grid(), _cover(units, 1)))
        want, _, _ = oracle.reduce_scatter("direct", xs, dtype)
        for r in range(n):
            g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "rs n=%d units=%d r=%d" % (n, units, r))
        del ins
        shards = [np.ascontiguousarray(x[:rc]) for x in xs]
        ins = [g.to_dev(x, dtype) for x in shards]
        outs = g.empty(n, n * rc, dtype)
        rra.rra_all_gather(ins, outs, rc, g.CODE[dtype], rra.RRA_ALGO_DIRECT)
        ag_grids.append((_last_grid(), _cover(units, 2)))
        want, _, _ = oracle.all_gather("direct", shards, dtype)
        for r in (0, n - 1):
            g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "ag n=%d units=%d r=%d" % (n, units, r))
        del ins, outs
    for grids in (rs_grids, ag_grids):
        (below, below_cover), (above, above_cover) = grids
        assert below != below_cover and above == above_cover, grids


@pytest.mark.parametrize("form", ["resident", "cover"])
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("n,rc", [(3, 100_003), (5, 4_097), (8, 1)])
def test_forced_grid_forms_match_oracle(form, dtype, n, rc, monkeypatch):
    # RRA_DIRECT_GRID forces one grid at every size: small and ragged
    # messages on the covering grid, and the resident one, give the
    # oracle's bits for all three operations
    g = G()
    monkeypatch.setenv("RRA_DIRECT_GRID", form)
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, n * rc, dtype, dist, seed=rc + n)
    ins = [g.to_dev(x, dtype) for x in xs]
    outs = g.empty(n, n * rc, dtype)
    rra.rra_allreduce(ins, outs, n * rc, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_ONE_SHOT)
    _last_grid()
    want, _, _ = oracle.allreduce("oneshot", xs, dtype)
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "one-shot %s r=%d" % (form, r))
    outs = g.empty(n, rc, dtype)
    rra.rra_reduce_scatter(ins, outs, rc, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_DIRECT)
    _last_grid()
    want, _, _ = oracle.reduce_scatter("direct", xs, dtype)
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "rs %s r=%d" % (form, r))
    shards = [np.ascontiguousarray(x[:rc]) for x in xs]
    ins = [g.to_dev(x, dtype) for x in shards]
    outs = g.empty(n, n * rc, dtype)
    rra.rra_all_gather(ins, outs, rc, g.CODE[dtype], rra.RRA_ALGO_DIRECT)
    _last_grid()
    want, _, _ = oracle.all_gather("direct", shards, dtype)
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], dtype), want[r], "ag %s r=%d" % (form, r))
