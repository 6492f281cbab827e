"""GPU path vs the CPU oracle at the largest sizes of the message-size
sweep, element by element, through the C ABI.

- n = 2, int32, 1 GiB per rank (the top of the sweep's x2 ladder, "Reading
  nccl-tests"), the size where an earlier sweep made AUTO choose the ring:
  the ring called directly, and AUTO against the oracle's result for the
  schedule it picks;
- n = 8, bfloat16, 256 MiB per rank, every all-reduce schedule;
- the literal one-shot form (RRA_ONESHOT_PER_RANK=1: each rank's CTAs read
  all n inputs, as n GPUs would) against the oracle's one-shot.

Inputs follow the sweep's recipe (inputs.cfg_sweep: int32 uniform in
[-2^20, 2^20], bfloat16 normal(0, 1), seeded).
"""
import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = pytest.mark.gpu

AR = {"ring": rra.RRA_ALGO_RING, "oneshot": rra.RRA_ALGO_ONE_SHOT, "twoshot": rra.RRA_ALGO_TWO_SHOT}


@pytest.fixture(scope="module", autouse=True)
def _init():
    import torch

    torch.cuda.set_device(0)
    rra.rra_init(0)
    rra.rra_set_timeout_ns(2_000_000_000)
    yield
    torch.cuda.empty_cache()


def _run(ins, outs, count, code, algo):
    rra.rra_allreduce(ins, outs, count, code, rra.RRA_SUM, algo)
    st, info = rra.rra_query_status()
    assert st == rra.RRA_SUCCESS, info


def test_ring_n2_int32_1gib_per_rank():
    import torch

    import gpu_util as g

    n, S = 2, 1 << 30
    xs = inputs.cfg_sweep(n, S, "int32", seed=S + n)
    count = xs[0].size
    want, _, _ = oracle.allreduce("ring", xs, "int32")
    ins = [g.to_dev(x, "int32") for x in xs]
    outs = g.empty(n, count, "int32")
    # AUTO runs whatever the shipped table picks at this size; int32 sums are
    # exact, so every schedule's result equals the ring's bit for bit
    picked = rra.rra_select_algo(n, S, rra.RRA_INT32)
    assert picked in (rra.RRA_ALGO_RING, rra.RRA_ALGO_ONE_SHOT, rra.RRA_ALGO_TWO_SHOT, rra.RRA_ALGO_TREE)
    for algo in (rra.RRA_ALGO_RING, rra.RRA_ALGO_AUTO):
        for o in outs:
            o.fill_(-0x5A5A5A5A)
        _run(ins, outs, count, rra.RRA_INT32, algo)
        for r in range(n):
            g.assert_bits_equal(g.to_host(outs[r], "int32"), want[r], "ring 1 GiB algo=%d r=%d" % (algo, r))
    del ins, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("algo", list(AR))
def test_n8_bf16_256mib_per_rank(algo):
    import torch

    import gpu_util as g

    n, S = 8, 256 << 20
    xs = inputs.cfg_sweep(n, S, "bfloat16", seed=S + n)
    count = xs[0].size
    want, _, _ = oracle.allreduce(algo, xs, "bfloat16")
    ins = [g.to_dev(x, "bfloat16") for x in xs]
    outs = g.empty(n, count, "bfloat16")
    _run(ins, outs, count, rra.RRA_BFLOAT16, AR[algo])
    for r in range(n):
        got = g.to_host(outs[r], "bfloat16")
        assert g.bf16_rel_ok(got, want[r]), (algo, r)
        g.assert_bits_equal(got, want[r], "%s bf16 256 MiB r=%d" % (algo, r))
    del ins, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,count", [(2, 5), (3, 4099), (8, 1_000_003), (8, 25_000_000 // 8 + 3)])
def test_oneshot_per_rank_form(dtype, n, count, monkeypatch):
    import gpu_util as g

    monkeypatch.setenv("RRA_ONESHOT_PER_RANK", "1")
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + n)
    want, _, _ = oracle.allreduce("oneshot", xs, dtype)
    # out of place: the literal form (in place keeps the combined form, which
    # reads a unit of every input before writing any output)
    for inplace in (False, True):
        ins = [g.to_dev(x, dtype) for x in xs]
        outs = ins if inplace else g.empty(n, count, dtype)
        _run(ins, outs, count, g.CODE[dtype], rra.RRA_ALGO_ONE_SHOT)
        for r in range(n):
            got = g.to_host(outs[r], dtype)
            if dtype == "bfloat16":
                assert g.bf16_rel_ok(got, want[r])
            g.assert_bits_equal(got, want[r], "one-shot per rank n=%d r=%d inplace=%s" % (n, r, inplace))
