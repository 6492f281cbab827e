"""The all-reduce entry point that allocates nothing.

Some callers may not allocate device memory: a plugin inside a framework
whose allocator owns the whole GPU, or code held to a memory budget after
start-up.  They cannot call rra_init, whose workspace comes from cudaMalloc.
rra_allreduce_two_shot_static gives them the two-shot all-reduce with its
scratch in a static device array inside the library.  These tests call it
through the C ABI twice in a row and compare each result with the regular
two-shot entry point's and with the oracle's two-shot, at the same bar as
the other parity tests: bit for bit, and for bfloat16 also within 1e-2
relative.  One test runs the entry point in a fresh process that never
calls rra_init, the case it exists for.

This file is collected last on purpose, and it passes both on its own in a
fresh process and after every other test.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    import torch

    torch.cuda.set_device(0)
    rra.rra_init(0)  # for the regular entry point the results are compared with
    yield


def _dev(x, dtype):
    import gpu_util

    return gpu_util.to_dev(x, dtype)


def _host(t, dtype):
    import gpu_util

    return gpu_util.to_host(t, dtype)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,count", [(2, 4096), (8, 1_000_003), (5, 77), (8, 25_000_000 // 4)])
def test_static_scratch_two_shot_matches_regular_entry_point(dtype, n, count):
    import torch

    import gpu_util

    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + n)
    ins = [_dev(x, dtype) for x in xs]
    code = gpu_util.CODE[dtype]

    want = gpu_util.empty(n, count, dtype)
    rra.rra_allreduce(ins, want, count, code, rra.RRA_SUM, rra.RRA_ALGO_TWO_SHOT)
    st, info = rra.rra_query_status()
    assert st == rra.RRA_SUCCESS, info
    ref = [_host(w, dtype) for w in want]
    if count <= 1_000_003:
        orc, _, _ = oracle.allreduce("twoshot", xs, dtype)
        for r in range(n):
            gpu_util.assert_bits_equal(ref[r], orc[r], "regular two-shot vs oracle, rank %d" % r)

    # first call on the device sets up the scratch address; later calls
    # must neither allocate nor change the result
    outs = [gpu_util.empty(n, count, dtype) for _ in range(2)]
    rra.rra_allreduce_two_shot_static(ins, outs[0], count, code)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for call in range(2):
        outs[call][0].fill_(0)
        rra.rra_allreduce_two_shot_static(ins, outs[call], count, code)
        torch.cuda.synchronize()
        for r in range(n):
            got = _host(outs[call][r], dtype)
            if dtype == "bfloat16":
                assert gpu_util.bf16_rel_ok(got, ref[r]), (call, r)
            gpu_util.assert_bits_equal(got, ref[r], "static call %d rank %d" % (call, r))
        st, info = rra.rra_query_status_static()
        assert st == rra.RRA_SUCCESS, info
    assert torch.cuda.mem_get_info()[0] == free_before


def test_static_scratch_in_place_and_errors():
    import torch

    import gpu_util

    n, count = 4, 300_001
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=4)
    ins = [_dev(x, "float32") for x in xs]
    want = gpu_util.empty(n, count, "float32")
    rra.rra_allreduce(ins, want, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TWO_SHOT)
    rra.rra_allreduce_two_shot_static(ins, ins, count, rra.RRA_FLOAT32)
    torch.cuda.synchronize()
    for r in range(n):
        gpu_util.assert_bits_equal(_host(ins[r], "float32"), _host(want[r], "float32"), "in place")
    # more ranks than the static flags hold, overlapping outputs, bad dtype
    A = 1 << 40
    assert rra.rra_allreduce_two_shot_static([A] * 9, [A] * 9, 16, rra.RRA_FLOAT32,
                                             check=False) == rra.RRA_ERR_UNSUPPORTED
    assert rra.rra_allreduce_two_shot_static([A, A + (1 << 30)], [A + (2 << 30), A + (2 << 30) + 8], 16,
                                             rra.RRA_FLOAT32, check=False) == rra.RRA_ERR_ALIAS
    assert rra.rra_allreduce_two_shot_static([A, A + (1 << 30)], [A + (2 << 30), A + (3 << 30)], 16, 9,
                                             check=False) == rra.RRA_ERR_INVALID_ARG
    assert rra.rra_allreduce_two_shot_static([A, A + (1 << 30)], [A + (2 << 30), A + (3 << 30)], 0,
                                             rra.RRA_FLOAT32, check=False) == rra.RRA_SUCCESS


_FRESH = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import collective_all_reduce_rank_gb300 as rra
import oracle
from collective_all_reduce_rank_gb300 import inputs

torch.cuda.set_device(0)
# no rra_init anywhere in this process: the regular entry point refuses
# the two-shot, the static one needs nothing
for dtype, code, dist in (("int32", rra.RRA_INT32, "int20"), ("float32", rra.RRA_FLOAT32, "normal")):
    n, count = 8, 1_000_003
    xs = inputs.make_ranks(n, count, dtype, dist, seed=11)
    ins = [torch.from_numpy(x).cuda() for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    st = rra.rra_allreduce(ins, outs, count, code, rra.RRA_SUM, rra.RRA_ALGO_TWO_SHOT, check=False)
    assert st == rra.RRA_ERR_NOT_INITIALIZED, st
    want, _, _ = oracle.allreduce("twoshot", xs, dtype)
    for call in range(2):
        for t in outs:
            t.zero_()
        rra.rra_allreduce_two_shot_static(ins, outs, count, code)
        st, info = rra.rra_query_status_static()
        assert st == rra.RRA_SUCCESS, (st, info)
        for r in range(n):
            assert outs[r].cpu().numpy().tobytes() == want[r].tobytes(), (dtype, call, r)
assert "allreduce_two_shot_static" in rra.rra_dump_recent()
print("fresh process ok")
"""


def test_static_scratch_in_a_process_that_never_calls_rra_init():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True, timeout=600)
    assert p.returncode == 0 and "fresh process ok" in p.stdout, p.stdout + p.stderr
