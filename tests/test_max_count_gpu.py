"""The largest counts: more than 2^31 elements per rank, so element indices
pass 2^31 and byte offsets pass 2^32 and 2^33 -- where a 32-bit index or
offset anywhere on the path would wrap.

Buffers this large are filled on the device with counter-based integers in
[-128, 128) (inputs.counter_ints); the host computes the same values for a
sample of indices: both ends, every chunk and half boundary, the indices
around 2^28, 2^29, 2^30 and 2^31 elements, the ragged tail, and seeded
random ones.  Every partial sum of such values is an integer of magnitude
at most 1024, exact in int32, float32 and bfloat16 alike, so every schedule
and order gives the same bits: the oracle (its one-shot, direct
reduce-scatter and all-gather) on the sampled indices is the expected value
for every schedule.  Summation orders are pinned by the other parity tests;
this one checks that every element lands where it belongs.
"""
import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FILL_CHUNK = 1 << 27  # elements per device fill step (1 GiB of int64 indices)


@pytest.fixture(scope="module", autouse=True)
def _init():
    import torch

    torch.cuda.set_device(0)
    rra.rra_init(0)
    rra.rra_set_timeout_ns(2_000_000_000)
    yield
    torch.cuda.empty_cache()


def _fill(t, rank, first=0):
    """t[i] = counter_ints(rank, first + i), on the device."""
    import torch

    for a in range(0, t.numel(), FILL_CHUNK):
        b = min(t.numel(), a + FILL_CHUNK)
        idx = torch.arange(first + a, first + b, dtype=torch.int64, device=t.device)
        t[a:b] = inputs.counter_ints(rank, idx).to(t.dtype)
        del idx


def _host(rank, idx, dtype):
    v = inputs.counter_ints(rank, idx.astype(np.int64))
    if dtype == "int32":
        return v.astype(np.int32)
    if dtype == "float32":
        return v.astype(np.float32)
    return inputs.to_bf16_bits(v.astype(np.float32))


def _sample(count, parts, dtype, seed):
    """Sorted unique indices in [0, count) around every place a wrap or an
    off-by-one would show."""
    b = oracle.chunk_plan(parts, count, dtype)
    marks = list(b) + [1 << 28, 1 << 29, 1 << 30, 1 << 31, count]
    if parts != 2:
        marks += list(oracle.chunk_plan(2, count, dtype))  # the tree's two halves
    pts = [np.arange(m - 64, m + 64) for m in marks]
    pts.append(np.arange(0, 256))
    pts.append(np.random.default_rng(seed).integers(0, count, 8192))
    idx = np.unique(np.concatenate(pts))
    return idx[(idx >= 0) & (idx < count)].astype(np.int64)


def _gather(t, idx, dtype):
    import torch

    import gpu_util as g

    return g.to_host(t[torch.from_numpy(idx).to(t.device)], dtype)


def _check_allreduce(outs, idx, want, n, dtype, what):
    import gpu_util as g

    for r in range(n):
        got = _gather(outs[r], idx, dtype)
        g.assert_bits_equal(got, want[r], "%s r=%d" % (what, r))


@pytest.mark.parametrize("dtype", ["int32", "float32"])
def test_allreduce_n2_more_than_2_31_elements(dtype):
    import torch

    import gpu_util as g

    n, count = 2, (1 << 31) + 4099
    idx = _sample(count, n, dtype, seed=count)
    want, _, _ = oracle.allreduce("oneshot", [_host(k, idx, dtype) for k in range(n)], dtype)
    ins = [torch.empty(count + 1, dtype=g.TORCH[dtype], device="cuda") for _ in range(n)]
    outs = [torch.empty(count + 1, dtype=g.TORCH[dtype], device="cuda") for _ in range(n)]
    for k in range(n):
        _fill(ins[k][:count], k)
    algos = [("ring", rra.RRA_ALGO_RING), ("oneshot", rra.RRA_ALGO_ONE_SHOT),
             ("twoshot", rra.RRA_ALGO_TWO_SHOT), ("tree", rra.RRA_ALGO_TREE), ("auto", rra.RRA_ALGO_AUTO)]
    for name, algo in algos:
        for o in outs:
            o.view(torch.int32).fill_(-1)
        rra.rra_allreduce([x[:count] for x in ins], [o[:count] for o in outs], count, g.CODE[dtype],
                          rra.RRA_SUM, algo)
        st, info = rra.rra_query_status()
        assert st == 0, (name, info)
        _check_allreduce([o[:count] for o in outs], idx, want, n, dtype, "%s %s" % (name, dtype))
    # buffers 4 bytes past a 16-byte boundary: the element-wise ring and one-shot
    for k in range(n):
        _fill(ins[k][1:], k)
    for name, algo in (("ring", rra.RRA_ALGO_RING), ("oneshot", rra.RRA_ALGO_ONE_SHOT)):
        rra.rra_allreduce([x[1:] for x in ins], [o[1:] for o in outs], count, g.CODE[dtype], rra.RRA_SUM, algo)
        st, info = rra.rra_query_status()
        assert st == 0, (name, info)
        _check_allreduce([o[1:] for o in outs], idx, want, n, dtype, "%s unaligned %s" % (name, dtype))
    # in place: the ring overwrites its inputs
    rra.rra_allreduce([x[1:] for x in ins], [x[1:] for x in ins], count, g.CODE[dtype], rra.RRA_SUM,
                      rra.RRA_ALGO_RING)
    st, info = rra.rra_query_status()
    assert st == 0, info
    _check_allreduce([x[1:] for x in ins], idx, want, n, dtype, "ring in place %s" % dtype)
    del ins, outs
    torch.cuda.empty_cache()


def test_allreduce_n8_bf16_more_than_2_31_elements():
    import torch

    import gpu_util as g

    n, count, dtype = 8, (1 << 31) + 5, "bfloat16"
    idx = _sample(count, n, dtype, seed=count)
    want, _, _ = oracle.allreduce("oneshot", [_host(k, idx, dtype) for k in range(n)], dtype)
    ins = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    outs = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    for k in range(n):
        _fill(ins[k], k)
    for name, algo in (("ring", rra.RRA_ALGO_RING), ("oneshot", rra.RRA_ALGO_ONE_SHOT),
                       ("twoshot", rra.RRA_ALGO_TWO_SHOT), ("tree", rra.RRA_ALGO_TREE)):
        for o in outs:
            o.view(torch.int16).fill_(-1)
        rra.rra_allreduce(ins, outs, count, rra.RRA_BFLOAT16, rra.RRA_SUM, algo)
        st, info = rra.rra_query_status()
        assert st == 0, (name, info)
        _check_allreduce(outs, idx, want, n, dtype, "%s bf16 n=8" % name)
    del ins, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("algo", ["ring", "direct"])
def test_reduce_scatter_and_all_gather_past_2_32_bytes(algo):
    import torch

    import gpu_util as g

    code = {"ring": rra.RRA_ALGO_RING, "direct": rra.RRA_ALGO_DIRECT}[algo]
    n, c, dtype = 2, (1 << 30) + 3, "int32"  # the reduce-scatter input: 2c elements (8 GiB) per rank
    j = _sample(c, 1, dtype, seed=c)
    # reduce-scatter: rank r's output element i sums element r*c + i of every input
    ins = [torch.empty(n * c, dtype=torch.int32, device="cuda") for _ in range(n)]
    for k in range(n):
        _fill(ins[k], k)
    outs = g.empty(n, c, dtype)
    rra.rra_reduce_scatter(ins, outs, c, rra.RRA_INT32, rra.RRA_SUM, code)
    st, info = rra.rra_query_status()
    assert st == 0, info
    sub = [np.concatenate([_host(k, q * c + j, dtype) for q in range(n)]) for k in range(n)]
    want, _, _ = oracle.reduce_scatter("direct", sub, dtype)
    for r in range(n):
        g.assert_bits_equal(_gather(outs[r], j, dtype), want[r], "RS %s r=%d" % (algo, r))
    del ins, outs
    torch.cuda.empty_cache()
    # all-gather: rank r's output element q*c + i is element i of rank q
    ins = [torch.empty(c, dtype=torch.int32, device="cuda") for _ in range(n)]
    for k in range(n):
        _fill(ins[k], k)
    outs = g.empty(n, n * c, dtype)
    rra.rra_all_gather(ins, outs, c, rra.RRA_INT32, code)
    st, info = rra.rra_query_status()
    assert st == 0, info
    want, _, _ = oracle.all_gather("direct", [_host(k, j, dtype) for k in range(n)], dtype)
    pos = np.concatenate([q * c + j for q in range(n)])
    for r in range(n):
        g.assert_bits_equal(_gather(outs[r], pos, dtype), want[r], "AG %s r=%d" % (algo, r))
    del ins, outs
    torch.cuda.empty_cache()
