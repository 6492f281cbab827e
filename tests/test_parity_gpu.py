"""GPU path vs the CPU oracle, element by element, through the C ABI.

The bar: bit-exact for int32 and for float32 (the kernels sum in the
oracle's order), and for bfloat16 the 1e-2 relative bound (with float32
accumulation in the same order the results are expected bit-exact too, and
the tests check both).
"""
import numpy as np
import pytest

import oracle
import collective_all_reduce_rank_gb300 as rra
from collective_all_reduce_rank_gb300 import inputs

pytestmark = pytest.mark.gpu

AR = {"ring": rra.RRA_ALGO_RING, "oneshot": rra.RRA_ALGO_ONE_SHOT, "twoshot": rra.RRA_ALGO_TWO_SHOT}
RSAG = {"ring": rra.RRA_ALGO_RING, "direct": rra.RRA_ALGO_DIRECT}


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


def _check(got, want, dtype, what):
    g = G()
    if dtype == "bfloat16":
        assert g.bf16_rel_ok(got, want), what
    g.assert_bits_equal(got, want, what)


def _status_ok():
    st, info = rra.rra_query_status()
    assert st == rra.RRA_SUCCESS, info


def run_allreduce(xs, dtype, algo, inplace=False, offset=0):
    g = G()
    n, count = len(xs), xs[0].size
    if offset:
        # element-aligned but not 16-byte aligned buffers: the element path
        big = [g.to_dev(np.concatenate([np.zeros(offset, x.dtype), x]), dtype) for x in xs]
        ins = [b[offset:] for b in big]
        outs_big = g.empty(n, count + offset, dtype)
        outs = [o[offset:] for o in outs_big]
    else:
        ins = [g.to_dev(x, dtype) for x in xs]
        outs = ins if inplace else g.empty(n, count, dtype)
    rra.rra_allreduce(ins, outs, count, g.CODE[dtype], rra.RRA_SUM, AR[algo])
    _status_ok()
    return [g.to_host(o, dtype) for o in outs]


# --------------------------------------------------------------------------


@pytest.mark.parametrize("algo", list(AR))
@pytest.mark.parametrize("n", [2, 4, 8])
@pytest.mark.parametrize("dtype", ["float32", "int32", "bfloat16"])
def test_all_ones_sanity(algo, n, dtype):
    xs = inputs.make_ranks(n, 128, dtype, "ones")
    got = run_allreduce(xs, dtype, algo)
    want, _, _ = oracle.allreduce(algo, xs, dtype)
    for r in range(n):
        _check(got[r], want[r], dtype, "ones r=%d" % r)
        vals = G().bf16_bits_to_f64(got[r]) if dtype == "bfloat16" else got[r]
        assert np.all(vals == n)


@pytest.mark.parametrize("algo", list(AR))
def test_small_exact_config(algo):
    # n=2, float32 integers in [-8, 8], 4096 per rank
    xs = inputs.cfg_small_exact()
    got = run_allreduce(xs, "float32", algo)
    want, _, _ = oracle.allreduce(algo, xs, "float32")
    for r in range(2):
        _check(got[r], want[r], "float32", "r=%d" % r)


@pytest.mark.parametrize("algo", list(RSAG))
def test_small_exact_config_rs_ag(algo):
    g = G()
    xs = inputs.cfg_small_exact()
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = g.empty(2, 2048, "float32")
    rra.rra_reduce_scatter(ins, outs, 2048, rra.RRA_FLOAT32, rra.RRA_SUM, RSAG[algo])
    _status_ok()
    want, _, _ = oracle.reduce_scatter(algo, xs, "float32")
    for r in range(2):
        _check(g.to_host(outs[r], "float32"), want[r], "float32", "rs r=%d" % r)
    shards = [x[:2048].copy() for x in xs]
    ins = [g.to_dev(x, "float32") for x in shards]
    outs = g.empty(2, 4096, "float32")
    rra.rra_all_gather(ins, outs, 2048, rra.RRA_FLOAT32, RSAG[algo])
    _status_ok()
    want, _, _ = oracle.all_gather(algo, shards, "float32")
    for r in range(2):
        _check(g.to_host(outs[r], "float32"), want[r], "float32", "ag r=%d" % r)


@pytest.mark.parametrize("algo", list(AR))
@pytest.mark.parametrize("tokens", inputs.TP_TOKENS)
def test_tp_activations_bf16(algo, tokens):
    xs = inputs.cfg_tp_activations(tokens)
    got = run_allreduce(xs, "bfloat16", algo)
    want, _, _ = oracle.allreduce(algo, xs, "bfloat16")
    for r in range(8):
        _check(got[r], want[r], "bfloat16", "tokens=%d r=%d" % (tokens, r))


@pytest.mark.parametrize("algo", list(AR))
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_order_sensitive_float_data(algo, dtype, n):
    # several tiles and channels, plus a ragged tail
    count = 3 * 1024 * 16 * n + 7 * 8 + 3
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=21 + n, sigma=1e-2 if dtype == "float32" else 1.0)
    got = run_allreduce(xs, dtype, algo)
    want, _, _ = oracle.allreduce(algo, xs, dtype)
    for r in range(n):
        _check(got[r], want[r], dtype, "%s n=%d r=%d" % (algo, n, r))


@pytest.mark.parametrize("path", ["cluster", "simple", "ll", "staged"])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,count", [(2, 3), (3, 1001), (5, 70_001), (8, 8 * 4096 * 6 + 5), (8, 2_000_000),
                                     (4, 3 * 2048 * 8 * 4)])
def test_ring_link_protocols(path, dtype, n, count, monkeypatch):
    # the ring on a thread-block cluster (links in distributed shared
    # memory), per-warp with Simple (fence + head flag) or LL (flag in every
    # line) links in L2, or with whole-CTA messages staged in shared memory:
    # same bits as the oracle's ring, for all three ring operations
    if path == "cluster":
        monkeypatch.setenv("RRA_RING_CLUSTER", "1")
    else:
        monkeypatch.setenv("RRA_RING_CLUSTER", "0")
        monkeypatch.setenv("RRA_RING_PROTO", path)
    g = G()
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + n)
    for rep in range(2):
        got = run_allreduce(xs, dtype, "ring")
        want, _, _ = oracle.allreduce("ring", xs, dtype)
        for r in range(n):
            _check(got[r], want[r], dtype, "%s ring n=%d r=%d rep=%d" % (path, n, r, rep))
    rc = max(1, count // n)
    xs = inputs.make_ranks(n, n * rc, dtype, dist, seed=rc)
    ins = [g.to_dev(x, dtype) for x in xs]
    outs = g.empty(n, rc, dtype)
    rra.rra_reduce_scatter(ins, outs, rc, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_RING)
    _status_ok()
    want, _, _ = oracle.reduce_scatter("ring", xs, dtype)
    for r in range(n):
        _check(g.to_host(outs[r], dtype), want[r], dtype, "%s ring rs r=%d" % (path, r))
    shards = [x[:rc].copy() for x in xs]
    ins = [g.to_dev(x, dtype) for x in shards]
    outs = g.empty(n, n * rc, dtype)
    rra.rra_all_gather(ins, outs, rc, g.CODE[dtype], rra.RRA_ALGO_RING)
    _status_ok()
    want, _, _ = oracle.all_gather("ring", shards, dtype)
    for r in range(n):
        _check(g.to_host(outs[r], dtype), want[r], dtype, "%s ring ag r=%d" % (path, r))


@pytest.mark.parametrize("tile,G,K,stages", [(1024, 8, 16, 8), (128, 1, 2, 1), (256, 3, 4, 2), (512, 8, 9, 3),
                                             (4096, 2, 3, 8), (2048, 4, 8, 3)])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,count", [(1, 1000), (2, 3), (3, 100_003), (8, 8 * 1024 * 8 * 19 + 7), (8, 3_000_001),
                                     (6, 4 * 4096 * 33)])
def test_ring_staged_shapes(tile, G, K, stages, dtype, n, count, monkeypatch):
    # the staged ring over message sizes, steps, FIFO depths and pipeline
    # depths, including the smallest (one slot of credit beyond G, one
    # stage) and fewer stages than slot loaders: same bits as the oracle's
    # ring, twice in a row (the second call reuses the link counters under a
    # new epoch), in place as well
    monkeypatch.setenv("RRA_RING_PROTO", "staged")
    monkeypatch.setenv("RRA_RING_CLUSTER", "0")
    for k, v in (("RRA_RING_TILE", tile), ("RRA_RING_G", G), ("RRA_RING_K", K), ("RRA_RING_STAGES", stages)):
        monkeypatch.setenv(k, str(v))
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + n + tile)
    want, _, _ = oracle.allreduce("ring", xs, dtype)
    for rep, inplace in enumerate((False, True)):
        got = run_allreduce(xs, dtype, "ring", inplace=inplace)
        for r in range(n):
            _check(got[r], want[r], dtype, "staged n=%d r=%d rep=%d" % (n, r, rep))


@pytest.mark.parametrize("tile,G,K,stages", [(1024, 8, 16, 8), (128, 1, 2, 1), (256, 3, 4, 2), (2048, 4, 8, 3)])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,rc", [(2, 4), (3, 33_336), (5, 4096 * 7), (8, 1024 * 8 * 19 + 4), (8, 375_000)])
def test_ring_staged_rs_ag_shapes(tile, G, K, stages, dtype, n, rc, monkeypatch):
    # the staged ring's reduce-scatter and all-gather halves over message
    # sizes, steps, FIFO depths and pipeline depths: the all-gather's
    # forwards and the reduce-scatter's last step are read from the
    # sender's output, not a FIFO slot; out of place and in place (the RS
    # output at slice r of rank r's input, the AG shard at slot r of rank
    # r's output)
    monkeypatch.setenv("RRA_RING_PROTO", "staged")
    monkeypatch.setenv("RRA_RING_CLUSTER", "0")
    for k, v in (("RRA_RING_TILE", tile), ("RRA_RING_G", G), ("RRA_RING_K", K), ("RRA_RING_STAGES", stages)):
        monkeypatch.setenv(k, str(v))
    import gpu_util as g

    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, n * rc, dtype, dist, seed=rc + n + tile)
    want, _, _ = oracle.reduce_scatter("ring", xs, dtype)
    for inplace in (False, True):
        ins = [g.to_dev(x, dtype) for x in xs]
        outs = [ins[r][r * rc:(r + 1) * rc] for r in range(n)] if inplace else g.empty(n, rc, dtype)
        rra.rra_reduce_scatter(ins, outs, rc, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_RING)
        _status_ok()
        for r in range(n):
            _check(g.to_host(outs[r], dtype), want[r], dtype, "staged rs n=%d r=%d inplace=%s" % (n, r, inplace))
    shards = [x[:rc].copy() for x in xs]
    want, _, _ = oracle.all_gather("ring", shards, dtype)
    for inplace in (False, True):
        outs = g.empty(n, n * rc, dtype)
        if inplace:
            for r in range(n):
                outs[r][r * rc:(r + 1) * rc].copy_(g.to_dev(shards[r], dtype))
            ins = [outs[r][r * rc:(r + 1) * rc] for r in range(n)]
        else:
            ins = [g.to_dev(x, dtype) for x in shards]
        rra.rra_all_gather(ins, outs, rc, g.CODE[dtype], rra.RRA_ALGO_RING)
        _status_ok()
        for r in range(n):
            _check(g.to_host(outs[r], dtype), want[r], dtype, "staged ag n=%d r=%d inplace=%s" % (n, r, inplace))


@pytest.mark.parametrize("cluster", ["0", "1"])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,count", [(2, 5), (3, 4099), (8, 8 * 2048 * 19 * 3 + 11), (8, 1_000_003), (7, 777_777)])
def test_two_shot_cluster_and_warp_forms(cluster, dtype, n, count, monkeypatch):
    # two-shot on a thread-block cluster (exchange through distributed
    # shared memory) and the per-warp form with flags in L2: same bits
    monkeypatch.setenv("RRA_TWOSHOT_CLUSTER", cluster)
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count)
    want, _, _ = oracle.allreduce("twoshot", xs, dtype)
    for inplace in (False, True):
        got = run_allreduce(xs, dtype, "twoshot", inplace=inplace)
        for r in range(n):
            _check(got[r], want[r], dtype, "cluster=%s n=%d r=%d inplace=%s" % (cluster, n, r, inplace))


@pytest.mark.parametrize("algo", list(AR))
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("count", [1, 3, 4, 5, 8, 9, 17, 31, 100, 1001, 65537])
def test_ragged_counts(algo, n, count):
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=count + n)
    got = run_allreduce(xs, "float32", algo)
    want, _, _ = oracle.allreduce(algo, xs, "float32")
    for r in range(n):
        _check(got[r], want[r], "float32", "n=%d count=%d r=%d" % (n, count, r))


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n", [1, 2, 3, 8])
@pytest.mark.parametrize("count", [4, 4099, 5 * 2048 * 4 + 13, 1_000_003])
def test_oneshot_bulk_copy_path(dtype, n, count, monkeypatch):
    # the bulk-copy (TMA) staged one-shot: same bits as the oracle's one-shot
    monkeypatch.setenv("RRA_ONESHOT_TMA", "1")
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=count + 7 * n)
    got = run_allreduce(xs, dtype, "oneshot")
    want, _, _ = oracle.allreduce("oneshot", xs, dtype)
    for r in range(n):
        _check(got[r], want[r], dtype, "tma n=%d count=%d r=%d" % (n, count, r))
    got = run_allreduce(xs, dtype, "oneshot", inplace=True)
    for r in range(n):
        _check(got[r], want[r], dtype, "tma in place r=%d" % r)


@pytest.mark.parametrize("algo", list(AR))
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_unaligned_element_path(algo, dtype):
    n, count = 4, 10_000 + 3
    xs = inputs.make_ranks(n, count, dtype, "normal", seed=5)
    got = run_allreduce(xs, dtype, algo, offset=1)
    want, _, _ = oracle.allreduce(algo, xs, dtype)
    for r in range(n):
        _check(got[r], want[r], dtype, "offset r=%d" % r)


@pytest.mark.parametrize("algo", list(AR))
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
def test_in_place(algo, dtype):
    n, count = 8, 200_003
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=8)
    got = run_allreduce(xs, dtype, algo, inplace=True)
    want, _, _ = oracle.allreduce(algo, xs, dtype)
    for r in range(n):
        _check(got[r], want[r], dtype, "inplace r=%d" % r)


def test_world_size_one_and_empty():
    g = G()
    xs = inputs.make_ranks(1, 1000, "float32", "normal")
    for algo in AR.values():
        assert run_allreduce(xs, "float32", [k for k, v in AR.items() if v == algo][0])[0].tobytes() == xs[0].tobytes()
    # count 0: success, no launch, outputs untouched
    ins = [g.to_dev(np.ones(4, np.float32), "float32") for _ in range(2)]
    outs = g.empty(2, 4, "float32", fill=7)
    rra.rra_allreduce(ins, outs, 0, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_RING)
    assert np.all(g.to_host(outs[0], "float32").view(np.int32) == 7)


@pytest.mark.parametrize("algo", list(RSAG))
@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n,rc", [(2, 2048), (3, 1001), (8, 5000), (8, 3), (5, 64 * 1024 + 1)])
def test_reduce_scatter_and_all_gather(algo, dtype, n, rc):
    g = G()
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, n * rc, dtype, dist, seed=rc)
    ins = [g.to_dev(x, dtype) for x in xs]
    outs = g.empty(n, rc, dtype)
    rra.rra_reduce_scatter(ins, outs, rc, g.CODE[dtype], rra.RRA_SUM, RSAG[algo])
    _status_ok()
    want, _, _ = oracle.reduce_scatter(algo, xs, dtype)
    for r in range(n):
        _check(g.to_host(outs[r], dtype), want[r], dtype, "rs r=%d" % r)
    shards = [x[:rc].copy() for x in xs]
    ins = [g.to_dev(x, dtype) for x in shards]
    outs = g.empty(n, n * rc, dtype)
    rra.rra_all_gather(ins, outs, rc, g.CODE[dtype], RSAG[algo])
    _status_ok()
    want, _, _ = oracle.all_gather(algo, shards, dtype)
    for r in range(n):
        _check(g.to_host(outs[r], dtype), want[r], dtype, "ag r=%d" % r)


@pytest.mark.parametrize("n,sc", [(2, 100), (8, 5000), (8, 3)])
def test_all_gather_copy_engine(n, sc):
    import torch

    g = G()
    shards = inputs.make_ranks(n, sc, "int32", "bits", seed=sc)
    ins = [g.to_dev(x, "int32") for x in shards]
    outs = g.empty(n, n * sc, "int32")
    rra.rra_all_gather(ins, outs, sc, rra.RRA_INT32, rra.RRA_ALGO_COPY_ENGINE)
    _status_ok()
    want, _, _ = oracle.all_gather("direct", shards, "int32")
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], "int32"), want[r], "copy engine r=%d" % r)
    # in place: shard r already at slot r of its own output
    bufs = [torch.zeros(n * sc, dtype=torch.int32, device="cuda") for _ in range(n)]
    for r in range(n):
        bufs[r][r * sc:(r + 1) * sc] = ins[r]
    rra.rra_all_gather([bufs[r][r * sc:(r + 1) * sc] for r in range(n)], bufs, sc, rra.RRA_INT32,
                       rra.RRA_ALGO_COPY_ENGINE)
    _status_ok()
    for r in range(n):
        g.assert_bits_equal(g.to_host(bufs[r], "int32"), want[r], "copy engine in place r=%d" % r)


@pytest.mark.parametrize("max_ctas", [1, 8, 19, 64])
def test_sm_budget_keeps_results(max_ctas):
    n, count = 8, 1_000_003
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=max_ctas)
    rra.rra_set_max_ctas(max_ctas)
    try:
        for algo in AR:
            got = run_allreduce(xs, "float32", algo)
            want, _, _ = oracle.allreduce(algo, xs, "float32")
            for r in (0, n - 1):
                _check(got[r], want[r], "float32", "%s max_ctas=%d" % (algo, max_ctas))
        text = rra.rra_dump_recent().strip().splitlines()[-1]
        assert "algo=two_shot" in text or "algo=ring" in text or "algo=one_shot" in text
    finally:
        rra.rra_set_max_ctas(0)


@pytest.mark.parametrize("algo", list(RSAG))
def test_rs_ag_in_place(algo):
    import torch

    g = G()
    n, rc = 4, 10_000
    xs = inputs.make_ranks(n, n * rc, "float32", "normal", seed=3)
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = [t[r * rc:(r + 1) * rc] for r, t in enumerate(ins)]
    rra.rra_reduce_scatter(ins, outs, rc, rra.RRA_FLOAT32, rra.RRA_SUM, RSAG[algo])
    _status_ok()
    want, _, _ = oracle.reduce_scatter(algo, xs, "float32")
    for r in range(n):
        _check(g.to_host(outs[r], "float32"), want[r], "float32", "rs in place r=%d" % r)
    bufs = [torch.zeros(n * rc, dtype=torch.float32, device="cuda") for _ in range(n)]
    shards = [x[:rc].copy() for x in xs]
    for r in range(n):
        bufs[r][r * rc:(r + 1) * rc] = g.to_dev(shards[r], "float32")
    ins = [bufs[r][r * rc:(r + 1) * rc] for r in range(n)]
    rra.rra_all_gather(ins, bufs, rc, rra.RRA_FLOAT32, RSAG[algo])
    _status_ok()
    want, _, _ = oracle.all_gather(algo, shards, "float32")
    for r in range(n):
        _check(g.to_host(bufs[r], "float32"), want[r], "float32", "ag in place r=%d" % r)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n", [2, 4, 8])
def test_ring_equals_rs_then_ag_on_gpu(dtype, n):
    g = G()
    rc = 4 * 1024 * 9
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, n * rc, dtype, dist, seed=77)
    ar = run_allreduce(xs, dtype, "ring")
    ins = [g.to_dev(x, dtype) for x in xs]
    mid = g.empty(n, rc, dtype)
    rra.rra_reduce_scatter(ins, mid, rc, g.CODE[dtype], rra.RRA_SUM, rra.RRA_ALGO_RING)
    outs = g.empty(n, n * rc, dtype)
    rra.rra_all_gather(mid, outs, rc, g.CODE[dtype], rra.RRA_ALGO_RING)
    _status_ok()
    for r in range(n):
        g.assert_bits_equal(g.to_host(outs[r], dtype), ar[r], "ring vs rs+ag r=%d" % r)


@pytest.mark.slow
@pytest.mark.parametrize("algo", list(AR))
def test_gradient_bucket_full_size(algo):
    # n=8, float32 normal(0, 1e-2), 25M elements per rank (100 MB): the full
    # workload the benchmark times, compared element by element.
    xs = inputs.cfg_gradient_bucket()
    got = run_allreduce(xs, "float32", algo)
    want, _, _ = oracle.allreduce(algo, xs, "float32")
    for r in range(8):
        _check(got[r], want[r], "float32", "bucket r=%d" % r)


def test_auto_and_repeat_calls_are_stable():
    # many calls in a row: the per-call epoch keeps the step flags apart
    g = G()
    n, count = 8, 300_000
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=9)
    ins = [g.to_dev(x, "float32") for x in xs]
    want = {a: oracle.allreduce(a, xs, "float32")[0] for a in AR}
    for rep in range(5):
        for a, code in AR.items():
            outs = g.empty(n, count, "float32")
            rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, code)
            _status_ok()
            for r in (0, n - 1):
                g.assert_bits_equal(g.to_host(outs[r], "float32"), want[a][r], "%s rep %d" % (a, rep))
    outs = g.empty(n, count, "float32")
    rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_AUTO)
    _status_ok()
    pick = rra.rra_select_algo(n, count * 4, rra.RRA_FLOAT32)
    name = {v: k for k, v in AR.items()}[pick]
    g.assert_bits_equal(g.to_host(outs[3], "float32"), want[name][3], "auto")


def test_cuda_graph_capture():
    import torch

    g = G()
    n, count = 4, 50_000
    xs = inputs.make_ranks(n, count, "float32", "normal", seed=10)
    ins = [g.to_dev(x, "float32") for x in xs]
    outs = g.empty(n, count, "float32")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, rra.RRA_ALGO_TWO_SHOT, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for a in (rra.RRA_ALGO_RING, rra.RRA_ALGO_TWO_SHOT, rra.RRA_ALGO_ONE_SHOT):
            rra.rra_allreduce(ins, outs, count, rra.RRA_FLOAT32, rra.RRA_SUM, a, stream=s)
    want, _, _ = oracle.allreduce("oneshot", xs, "float32")
    for rep in range(3):
        for o in outs:
            o.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        _status_ok()
        for r in range(n):
            g.assert_bits_equal(g.to_host(outs[r], "float32"), want[r], "graph replay %d" % rep)


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
@pytest.mark.parametrize("tokens", inputs.TP_TOKENS)
@pytest.mark.parametrize("n", [2, 8])
def test_allreduce_rmsnorm(dtype, tokens, n):
    # fused all-reduce + RMSNorm on [tokens, 5120]: within the 1e-2 relative
    # bar of the oracle (float64 normalisation of the float32 sums)
    g = G()
    hidden = inputs.TP_HIDDEN
    xs = inputs.make_ranks(n, tokens * hidden, dtype, "normal", seed=tokens + n)
    gamma = inputs.make_ranks(1, hidden, dtype, "normal", seed=99)[0]
    ins = [g.to_dev(x, dtype) for x in xs]
    outs = g.empty(n, tokens * hidden, dtype)
    rra.rra_allreduce_rmsnorm(ins, outs, g.to_dev(gamma, dtype), hidden, eps=1e-6)
    _status_ok()
    want = oracle.allreduce_rmsnorm(xs, gamma, 1e-6, dtype, hidden)
    for r in range(n):
        got = g.to_host(outs[r], dtype)
        if dtype == "bfloat16":
            assert g.bf16_rel_ok(got, want[r]), r
        else:
            w = want[r].astype(np.float64)
            assert np.all(np.abs(got.astype(np.float64) - w) <= 1e-5 * np.abs(w) + 1e-6), r
        assert got.tobytes() == g.to_host(outs[0], dtype).tobytes()


@pytest.mark.parametrize("hidden", [1, 7, 100, 4096, 12345])
def test_allreduce_rmsnorm_odd_rows_and_in_place(hidden):
    g = G()
    n, rows = 3, 5
    xs = inputs.make_ranks(n, rows * hidden, "float32", "normal", seed=hidden)
    gamma = inputs.make_ranks(1, hidden, "float32", "normal", seed=1)[0]
    ins = [g.to_dev(x, "float32") for x in xs]
    rra.rra_allreduce_rmsnorm(ins, ins, g.to_dev(gamma, "float32"), hidden, eps=1e-5)
    _status_ok()
    want = oracle.allreduce_rmsnorm(xs, gamma, 1e-5, "float32", hidden)
    for r in range(n):
        got = g.to_host(ins[r], "float32").astype(np.float64)
        w = want[r].astype(np.float64)
        assert np.all(np.abs(got - w) <= 1e-5 * np.abs(w) + 1e-6)
