"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test names what pins it: the pages' printed values (golden files), a
closed form, brute force in exact integer or double arithmetic, a library
routine (torch's bfloat16 cast), or a hand-derived value whose derivation is
written next to it.  Summation-order pins use values whose float32 sums
differ between orders, so a wrong rotation, a wrong starting rank or a
re-rounded bfloat16 partial fails one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import model
from collective_all_reduce_rank_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
AR_ALGOS = ("ring", "oneshot", "twoshot")
U32 = 2.0 ** -24  # float32 unit roundoff


def _gamma(k):
    return k * U32 / (1 - k * U32)


# --------------------------------------------------------------------------
# sanity test and world_size == 1


@pytest.mark.parametrize("n", [2, 3, 4, 8])
@pytest.mark.parametrize("algo", AR_ALGOS)
@pytest.mark.parametrize("dtype", ["float32", "int32", "bfloat16"])
def test_all_ones_sums_to_n(n, algo, dtype):
    # NCCL collectives ... "Code": an all-reduce of ones(128) gives world_size.
    xs = inputs.make_ranks(n, 128, dtype, "ones")
    outs, _, _ = oracle.allreduce(algo, xs, dtype)
    for o in outs:
        vals = oracle.bf16_to_f32(o) if dtype == "bfloat16" else o
        assert np.all(vals == n)


@pytest.mark.parametrize("algo", AR_ALGOS)
def test_world_size_one_is_identity(algo):
    # "bare python -> world_size == 1 -> tests nothing": the op is a no-op.
    for dtype in ("float32", "int32", "bfloat16"):
        xs = inputs.make_ranks(1, 1000, dtype, "normal" if dtype != "int32" else "int20")
        outs, sent, recv = oracle.allreduce(algo, xs, dtype)
        assert outs[0].tobytes() == xs[0].tobytes()
        assert sent == [0] and recv == [0]


# --------------------------------------------------------------------------
# brute force: exact sums


def _exact_int32_sum(xs):
    s = np.zeros(xs[0].size, dtype=np.int64)
    for x in xs:
        s += x.astype(np.int64)
    return ((s + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("count", [0, 1, 3, 4, 5, 17, 64, 1001])
def test_int32_brute_force_with_wraparound(n, count):
    xs = inputs.make_ranks(n, count, "int32", "bits", seed=n * 1000 + count)
    want = _exact_int32_sum(xs)
    for algo in AR_ALGOS:
        outs, _, _ = oracle.allreduce(algo, xs, "int32")
        for o in outs:
            assert np.array_equal(o, want), algo


def test_float32_integer_config_is_exact():
    # n=2, integers in [-8, 8]: every partial sum is exact in float32, so all
    # schedules must equal the exact (double) sum.
    xs = inputs.cfg_small_exact()
    want = (xs[0].astype(np.float64) + xs[1].astype(np.float64)).astype(np.float32)
    for algo in AR_ALGOS:
        outs, _, _ = oracle.allreduce(algo, xs, "float32")
        for o in outs:
            assert np.array_equal(o, want)


@pytest.mark.parametrize("n", [2, 3, 4, 7, 8])
def test_rs_ag_brute_force_int32(n):
    rc = 13
    xs = inputs.make_ranks(n, n * rc, "int32", "bits", seed=7 + n)
    total = _exact_int32_sum(xs)
    for algo in ("ring", "direct"):
        outs, _, _ = oracle.reduce_scatter(algo, xs, "int32")
        for r, o in enumerate(outs):
            assert np.array_equal(o, total[r * rc:(r + 1) * rc]), algo
    shards = inputs.make_ranks(n, rc, "int32", "bits", seed=99 + n)
    cat = np.concatenate(shards)
    for algo in ("ring", "direct"):
        outs, _, _ = oracle.all_gather(algo, shards, "int32")
        for o in outs:
            assert np.array_equal(o, cat), algo


# --------------------------------------------------------------------------
# summation order, pinned by hand-derived float32 values

B25 = float(2 ** 25)  # float32 spacing is 4 just above 2^25 and 2 just below


def _order_case():
    """n = 4, float32, count = 16 -> chunk plan gives four chunks of 4.

    In chunk c the ranks hold: x_{c+1} = 2^25, x_{c+2} = -2^25, x_{c+3} = 1,
    x_c = 0.5 (indices mod 4).  Derivations (float32, round to nearest):

    ring, order x_{c+1}, x_{c+2}, x_{c+3}, x_c:
        ((2^25 - 2^25) + 1) + 0.5 = 1.5 in every chunk.
    ascending rank order 0..3 (one-shot, two-shot), per chunk:
      c=0: x0=0.5, x1=2^25, x2=-2^25, x3=1:  (0.5+2^25) = 2^25 -> 0 -> 1
      c=1: x0=1, x1=0.5, x2=2^25, x3=-2^25:  1.5 + 2^25 = 2^25 -> 0
      c=2: x0=-2^25, x1=1, x2=0.5, x3=2^25:  -2^25+1 = -2^25 (tie to even)
                                             -> -2^25 + 0.5 = -2^25 -> 0
      c=3: x0=2^25, x1=-2^25, x2=1, x3=0.5:  0 + 1 + 0.5 = 1.5
    A ring turning the other way, x_{c-1}, x_{c-2}, x_{c-3}, x_c, gives
    ((1 - 2^25) + 2^25) + 0.5 = 0.5; a ring starting at its own rank gives
    ((0.5 + 2^25) - 2^25) + 1 = 1.
    """
    n, chunk = 4, 4
    xs = [np.zeros(n * chunk, dtype=np.float32) for _ in range(n)]
    for c in range(n):
        sl = slice(c * chunk, (c + 1) * chunk)
        xs[(c + 1) % n][sl] = B25
        xs[(c + 2) % n][sl] = -B25
        xs[(c + 3) % n][sl] = 1.0
        xs[c][sl] = 0.5
    return xs


def test_ring_summation_order_pinned():
    xs = _order_case()
    assert oracle.chunk_plan(4, 16, "float32") == [0, 4, 8, 12, 16]
    outs, _, _ = oracle.allreduce("ring", xs, "float32")
    for o in outs:
        assert np.array_equal(o, np.full(16, 1.5, np.float32))


@pytest.mark.parametrize("algo", ["oneshot", "twoshot"])
def test_ascending_summation_order_pinned(algo):
    xs = _order_case()
    want = np.repeat(np.array([1.0, 0.0, 0.0, 1.5], np.float32), 4)
    outs, _, _ = oracle.allreduce(algo, xs, "float32")
    for o in outs:
        assert np.array_equal(o, want)


def test_reduce_scatter_orders_pinned():
    xs = _order_case()  # 16 elements = 4 slices of rc = 4
    outs, _, _ = oracle.reduce_scatter("ring", xs, "float32")
    for o in outs:
        assert np.array_equal(o, np.full(4, 1.5, np.float32))
    outs, _, _ = oracle.reduce_scatter("direct", xs, "float32")
    for r, o in enumerate(outs):
        assert np.array_equal(o, np.full(4, [1.0, 0.0, 0.0, 1.5][r], np.float32))


def test_bf16_rounds_once_at_the_end():
    # bfloat16 of 1 has spacing 2^-7.  1 + 7 * 2^-9 = 1.013671875 is exact in
    # float32 and rounds to 1 + 2^-6 = 1.015625 in bfloat16.  Re-rounding each
    # partial to bfloat16 would keep 1 (2^-9 is a quarter of an ulp).
    n = 8
    vals = [1.0] + [2.0 ** -9] * 7
    xs = [inputs.to_bf16_bits(np.full(16, v, np.float32)) for v in vals]
    for algo in AR_ALGOS:
        outs, _, _ = oracle.allreduce(algo, xs, "bfloat16")
        for o in outs:
            assert np.all(oracle.bf16_to_f32(o) == np.float32(1.015625)), algo


# --------------------------------------------------------------------------
# error bounds for order-dependent float data


@pytest.mark.parametrize("algo", AR_ALGOS)
def test_float32_recursive_summation_bound(algo):
    # Higham's bound for recursive summation of n terms in any order:
    # |fl(sum) - sum| <= gamma_{n-1} * sum |x_k|.
    n = 8
    xs = inputs.make_ranks(n, 20_000, "float32", "normal", seed=3, sigma=1e-2)
    x64 = np.stack([x.astype(np.float64) for x in xs])
    exact = x64.sum(axis=0)
    absum = np.abs(x64).sum(axis=0)
    outs, _, _ = oracle.allreduce(algo, xs, "float32")
    for o in outs:
        assert np.all(np.abs(o.astype(np.float64) - exact) <= _gamma(n - 1) * absum)


@pytest.mark.parametrize("algo", AR_ALGOS)
def test_bf16_error_bound(algo):
    # out = RNE_bf16(s) with s the float32 sum: |RNE(s) - s| <= 2^-8 |s| and
    # |s - sum| <= gamma_{n-1} sum|x|, hence
    # |out - sum| <= 2^-8 (|sum| + g) + g,  g = gamma_{n-1} sum|x|.
    n = 8
    xs = inputs.make_ranks(n, 20_000, "bfloat16", "normal", seed=4)
    x64 = np.stack([oracle.bf16_to_f32(x).astype(np.float64) for x in xs])
    exact = x64.sum(axis=0)
    g = _gamma(n - 1) * np.abs(x64).sum(axis=0)
    bound = 2.0 ** -8 * (np.abs(exact) + g) + g
    outs, _, _ = oracle.allreduce(algo, xs, "bfloat16")
    for o in outs:
        got = oracle.bf16_to_f32(o).astype(np.float64)
        assert np.all(np.abs(got - exact) <= bound)
    # and nearly always the correctly rounded exact sum
    same = np.mean(oracle.bf16_to_f32(outs[0]) ==
                   oracle.bf16_to_f32(inputs.to_bf16_bits(exact.astype(np.float32))))
    assert same > 0.99


def test_bf16_rounding_matches_torch():
    # torch's float32 -> bfloat16 cast on the CPU rounds to nearest even.
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=20_000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF,
                        0x00000001, 0x00008000, 0x00018000, 0x3F808000, 0x3F818000,
                        0x3F80FFFF, 0x3F807FFF, 0x007FFFFF, 0xFF7FFFFF], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    f = bits.view(np.float32)
    finite = ~np.isnan(f)
    got = oracle.f32_to_bf16(f[finite])
    want = inputs.to_bf16_bits(f[finite])
    assert np.array_equal(got, want)
    # NaN stays NaN (the bit pattern of the NaN is not compared)
    nans = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0x7FFFFFFF], np.uint32).view(np.float32)
    assert np.all(np.isnan(oracle.bf16_to_f32(oracle.f32_to_bf16(nans))))


# --------------------------------------------------------------------------
# schedules as schedules: traffic closed forms


@pytest.mark.parametrize("n", [2, 3, 4, 8])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_per_rank_traffic_closed_forms(n, dtype):
    e = inputs.ELEM_SIZE[dtype]
    v = 16 // e
    count = n * v * 5
    S = count * e
    xs = inputs.make_ranks(n, count, dtype, "normal", seed=n)
    # ring: each GPU sends and receives 2(n-1)/n S
    _, sent, recv = oracle.allreduce("ring", xs, dtype)
    assert sent == recv == [2 * (n - 1) * S // n] * n
    # two-shot: reads 2(n-1)/n S per GPU
    _, sent, recv = oracle.allreduce("twoshot", xs, dtype)
    assert recv == [2 * (n - 1) * S // n] * n
    # one-shot: reads (n-1) S per GPU
    _, sent, recv = oracle.allreduce("oneshot", xs, dtype)
    assert recv == [(n - 1) * S] * n
    # reduce-scatter / all-gather: (n-1)/n of the per-rank input / output
    for algo in ("ring", "direct"):
        _, sent, recv = oracle.reduce_scatter(algo, xs, dtype)
        assert recv == [(n - 1) * S // n] * n
        shards = [x[: count // n].copy() for x in xs]
        _, sent, recv = oracle.all_gather(algo, shards, dtype)
        assert recv == [(n - 1) * S // n] * n


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("n", [2, 3, 8])
def test_ring_is_reduce_scatter_then_all_gather(dtype, n):
    # "Ring all-reduce = reduce-scatter + all-gather": bitwise, when count/n
    # is a whole number of 16-byte vectors (then the chunk plan's chunks are
    # exactly the reduce-scatter slices).
    v = 16 // inputs.ELEM_SIZE[dtype]
    count = n * v * 9
    dist = "int20" if dtype == "int32" else "normal"
    xs = inputs.make_ranks(n, count, dtype, dist, seed=11)
    ar, _, _ = oracle.allreduce("ring", xs, dtype)
    rs, _, _ = oracle.reduce_scatter("ring", xs, dtype)
    ag, _, _ = oracle.all_gather("ring", rs, dtype)
    for a, b in zip(ar, ag):
        assert a.tobytes() == b.tobytes()
    ar2, _, _ = oracle.allreduce("twoshot", xs, dtype)
    rs2, _, _ = oracle.reduce_scatter("direct", xs, dtype)
    ag2, _, _ = oracle.all_gather("direct", rs2, dtype)
    for a, b in zip(ar2, ag2):
        assert a.tobytes() == b.tobytes()


def test_oneshot_equals_twoshot_bitwise():
    # both sum in ascending rank order, element by element
    xs = inputs.make_ranks(8, 5000, "float32", "normal", seed=12, sigma=1e-2)
    a, _, _ = oracle.allreduce("oneshot", xs, "float32")
    b, _, _ = oracle.allreduce("twoshot", xs, "float32")
    for x, y in zip(a, b):
        assert x.tobytes() == y.tobytes()


# --------------------------------------------------------------------------
# chunk plan


def test_chunk_plan_examples():
    assert oracle.chunk_plan(2, 4096, "float32") == [0, 2048, 4096]
    b = oracle.chunk_plan(8, 25_000_000, "float32")
    assert b[1] == 3_125_000 and b[-1] == 25_000_000
    for t in inputs.TP_TOKENS:
        b = oracle.chunk_plan(8, t * 5120, "bfloat16")
        assert b[1] == 640 * t
    # ragged: count 10, n 4, float32 (V = 4): ceil(10/4) = 3 -> C = 4
    assert oracle.chunk_plan(4, 10, "float32") == [0, 4, 8, 10, 10]
    assert oracle.chunk_plan(3, 0, "int32") == [0, 0, 0, 0]


@pytest.mark.parametrize("n,count", [(3, 10), (4, 10), (8, 7), (5, 1), (7, 1000)])
def test_ragged_counts_all_schedules_exact(n, count):
    xs = inputs.make_ranks(n, count, "int32", "bits", seed=count)
    want = _exact_int32_sum(xs)
    for algo in AR_ALGOS:
        outs, _, _ = oracle.allreduce(algo, xs, "int32")
        for o in outs:
            assert np.array_equal(o, want)


# --------------------------------------------------------------------------
# LL / LL128


def _read_ll_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "ll_lines.txt"))
            if l.strip() and not l.startswith("#")]
    return rows


def test_ll_layout_golden():
    rows = _read_ll_golden()
    payload = bytes.fromhex(rows[0][1].split("=")[1])
    flag = int(rows[0][2].split("=")[1], 16)
    wire = bytes.fromhex(rows[1][1].split("=")[1])
    got = oracle.ll_pack(np.frombuffer(payload, np.uint8), flag)
    assert got.tobytes() == wire


def test_ll128_layout_golden():
    rows = _read_ll_golden()
    flag = int(rows[2][2].split("=")[1], 16)
    payload = np.arange(130, dtype=np.uint8)
    got = oracle.ll128_pack(payload, flag).tobytes()
    fbytes = flag.to_bytes(8, "little")
    want = bytes(range(120)) + fbytes + bytes(range(120, 130)) + bytes(110) + fbytes
    assert got == want


@pytest.mark.parametrize("B", [4, 8, 12, 1024, 4000])
def test_protocol_efficiency(B):
    # LL: 4 data bytes per 8-byte line -> 50%; LL128: 120 per 128 -> 93.75%
    assert oracle.ll_wire_bytes(B) == 8 * math.ceil(B / 4)
    assert oracle.ll128_wire_bytes(B) == 128 * math.ceil(B / 120)
    assert B / oracle.ll_wire_bytes(B) == 0.5
    assert oracle.ll128_wire_bytes(120 * B) == 128 * B
    assert 120 * B / oracle.ll128_wire_bytes(120 * B) == 0.9375


@pytest.mark.parametrize("fmt", ["ll", "ll128"])
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("B", [2, 4, 6, 118, 120, 122, 240, 1000, 4096])
def test_pack_unpack_identity(fmt, dtype, B):
    e = inputs.ELEM_SIZE[dtype]
    if B % e:
        pytest.skip("payload must be whole elements")
    dist = "int20" if dtype == "int32" else "normal"
    x = inputs.make_ranks(1, B // e, dtype, dist, seed=B)[0]
    pack = oracle.ll_pack if fmt == "ll" else oracle.ll128_pack
    unpack = oracle.ll_unpack if fmt == "ll" else oracle.ll128_unpack
    wire = pack(x, 3)
    out, bad = unpack([wire], B, dtype, 3)
    assert bad == -1
    assert out.tobytes() == x.tobytes()


@pytest.mark.parametrize("fmt", ["ll", "ll128"])
def test_unpack_reduce_int32_equals_allreduce(fmt):
    B = 4 * 3001
    xs = inputs.cfg_ll_payloads(B)
    pack = oracle.ll_pack if fmt == "ll" else oracle.ll128_pack
    unpack = oracle.ll_unpack if fmt == "ll" else oracle.ll128_unpack
    wires = [pack(x, 5) for x in xs]
    out, bad = unpack(wires, B, "int32", 5)
    assert bad == -1
    assert np.array_equal(out, _exact_int32_sum(xs))


@pytest.mark.parametrize("fmt", ["ll", "ll128"])
def test_unpack_float32_sums_sources_in_ascending_order(fmt):
    # sources 0..3 hold 2^25, -2^25, 1, 0.5: ascending gives 1.5; descending
    # would give ((0.5 + 1) - 2^25) + 2^25 = 2 (1.5 - 2^25 rounds to -2^25 + 2).
    vals = [B25, -B25, 1.0, 0.5]
    pack = oracle.ll_pack if fmt == "ll" else oracle.ll128_pack
    unpack = oracle.ll_unpack if fmt == "ll" else oracle.ll128_unpack
    wires = [pack(np.full(60, v, np.float32), 1) for v in vals]
    out, bad = unpack(wires, 240, "float32", 1)
    assert bad == -1 and np.all(out == 1.5)


@pytest.mark.parametrize("fmt", ["ll", "ll128"])
def test_unpack_reports_first_bad_flag(fmt):
    B = 4 * 12000
    xs = inputs.cfg_ll_payloads(B)
    pack = oracle.ll_pack if fmt == "ll" else oracle.ll128_pack
    unpack = oracle.ll_unpack if fmt == "ll" else oracle.ll128_unpack
    line, flag_off = (8, 4) if fmt == "ll" else (128, 120)
    wires = [pack(x, 7) for x in xs]
    # a call made one step late sees flags of the previous step everywhere
    _, bad = unpack(wires, B, "int32", 8)
    assert bad == 0
    # one corrupted flag in source 2, line 37
    wires[2][37 * line + flag_off] ^= 0x40
    _, bad = unpack(wires, B, "int32", 7)
    assert bad == 37


# --------------------------------------------------------------------------
# cost model and metrics: the pages' printed numbers


def _golden_table():
    rows, ring = [], None
    for l in open(os.path.join(GOLDEN, "alpha_beta_table.txt")):
        if not l.strip() or l.startswith("#"):
            continue
        p = l.split()
        if p[0] == "ring_1GiB":
            ring = tuple(float(v) for v in p[1:])
        else:
            rows.append((int(p[0]), [float(v) for v in p[1:6]], p[6]))
    return rows, ring


def test_alpha_beta_table_reproduced():
    rows, ring = _golden_table()
    assert len(rows) == 5
    for S, printed, best in rows:
        got = [model.ab_time(a, 8, S, 1.5e-6, 450e9) * 1e6 for a in model.ALGOS]
        assert [round(g, 1) for g in got] == printed
        fastest = min((a for a in model.ALGOS if a != "NVLS"),
                      key=lambda a: model.ab_time(a, 8, S, 1.5e-6, 450e9))
        assert fastest == best
    S = 1 << 30
    t = model.ab_time("ring", 8, S, 1.5e-6, 450e9)
    assert round(t * 1e3, 2) == ring[0]
    assert round(model.algbw(S, t) / 1e9) == ring[1]
    assert round(model.busbw("allreduce", 8, S, t) / 1e9) == ring[2]


def _golden_ex():
    d = {}
    for l in open(os.path.join(GOLDEN, "exercises.txt")):
        if l.strip() and not l.startswith("#"):
            k, v = l.split()
            d[k] = float(v)
    return d


def test_exercise_busbw_to_time():
    g = _golden_ex()
    n, busbw = 8, 360e9
    S = 256 * 2 ** 20
    ar_alg = busbw / model.bus_factor("allreduce", n)
    ag_alg = busbw / model.bus_factor("allgather", n)
    assert round(ar_alg / 1e9, 1) == g["ex1_allreduce_algbw_GBps"]
    assert round(S / ar_alg * 1e3, 1) == g["ex1_allreduce_ms"]
    assert round(ag_alg / 1e9) == g["ex1_allgather_algbw_GBps"]
    assert round(S / ag_alg * 1e3, 2) == g["ex1_allgather_ms"]
    assert model.bus_factor("reducescatter", n) == model.bus_factor("allgather", n) == 7 / 8
    assert model.bus_factor("broadcast", n) == 1.0


def test_crossover():
    g = _golden_ex()
    s8 = model.oneshot_twoshot_crossover(8, 1.5e-6, 450e9)
    assert round(s8 / 1e3) == g["ex2_crossover_n8_KB"]
    # at S* the two costs agree; below it one-shot wins, above it two-shot
    one = model.ab_time("one-shot", 8, s8, 1.5e-6, 450e9)
    two = model.ab_time("two-shot", 8, s8, 1.5e-6, 450e9)
    assert abs(one - two) < 1e-15
    assert model.oneshot_twoshot_crossover(2, 1.5e-6, 450e9) is None
    for S in (1e3, 1e6, 1e9):
        assert model.ab_time("one-shot", 2, S, 1.5e-6, 450e9) <= model.ab_time("two-shot", 2, S, 1.5e-6, 450e9)


# --------------------------------------------------------------------------
# fused all-reduce + RMSNorm


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_rmsnorm_matches_torch_float64(dtype):
    # library routine: torch's rms_norm in float64 on the float32 sums
    import torch

    n, rows, hidden, eps = 4, 6, 5120, 1e-6
    xs = inputs.make_ranks(n, rows * hidden, dtype, "normal", seed=31)
    gamma = inputs.make_ranks(1, hidden, dtype, "normal", seed=32)[0]
    outs = oracle.allreduce_rmsnorm(xs, gamma, eps, dtype, hidden)
    sums, _, _ = oracle.allreduce("oneshot", xs, dtype)
    # the oracle's float32 sums, recovered exactly for float32; for bfloat16
    # recompute them in float32 from the widened inputs (same order)
    if dtype == "float32":
        s = torch.from_numpy(sums[0].astype(np.float64)).view(rows, hidden)
        g = torch.from_numpy(gamma.astype(np.float64))
    else:
        acc = np.zeros(rows * hidden, np.float32)
        for x in xs:
            acc = acc + oracle.bf16_to_f32(x)
        s = torch.from_numpy(acc.astype(np.float64)).view(rows, hidden)
        g = torch.from_numpy(oracle.bf16_to_f32(gamma).astype(np.float64))
    want = torch.nn.functional.rms_norm(s, (hidden,), weight=g, eps=eps).reshape(-1).numpy()
    for o in outs:
        got = o.astype(np.float64) if dtype == "float32" else oracle.bf16_to_f32(o).astype(np.float64)
        ulp = 2.0 ** -23 if dtype == "float32" else 2.0 ** -7
        assert np.all(np.abs(got - want) <= ulp * np.abs(want) + 1e-30)
    assert all(o.tobytes() == outs[0].tobytes() for o in outs)


def test_rmsnorm_closed_forms():
    # a row of equal sums c gives gamma * c / sqrt(c^2 + eps); eps = 0 -> gamma
    n, hidden = 2, 64
    xs = [np.full(2 * hidden, 1.5, np.float32), np.full(2 * hidden, 2.0, np.float32)]
    gamma = np.linspace(-2, 2, hidden).astype(np.float32)
    out = oracle.allreduce_rmsnorm(xs, gamma, 0.0, "float32", hidden)[0]
    assert np.allclose(out, np.tile(gamma, 2), rtol=0, atol=2e-7)
    out = oracle.allreduce_rmsnorm(xs, gamma, 3.0, "float32", hidden)[0]
    want = gamma.astype(np.float64) * 3.5 / np.sqrt(3.5 ** 2 + 3.0)
    assert np.allclose(out, np.tile(want, 2), rtol=1e-7, atol=0)
    # scale invariance with eps = 0 and the unit mean square of the output
    xs = inputs.make_ranks(3, 4 * hidden, "float32", "normal", seed=2)
    a = oracle.allreduce_rmsnorm(xs, np.ones(hidden, np.float32), 0.0, "float32", hidden)[0]
    b = oracle.allreduce_rmsnorm([x * 8 for x in xs], np.ones(hidden, np.float32), 0.0, "float32", hidden)[0]
    assert np.array_equal(a, b)  # power-of-two scaling is exact
    ms = (a.astype(np.float64).reshape(4, hidden) ** 2).mean(axis=1)
    assert np.allclose(ms, 1.0, rtol=1e-6)
