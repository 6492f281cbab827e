"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad arguments synchronously, before any launch."""
import ctypes
import math
import os

import pytest

import collective_all_reduce_rank_gb300 as rra


@pytest.fixture(scope="module")
def lib():
    return rra.load()


def test_exports_every_declared_symbol(lib):
    names = rra.header_symbols()
    assert len(names) >= 18
    for name in names:
        assert hasattr(lib, name), name
    # nothing from the oracle leaks into the product library
    out = os.popen("nm -D --defined-only %s" % rra.library_path()).read()
    assert "orc_" not in out


def test_status_strings(lib):
    for code in range(8):
        assert rra.rra_status_string(code) != "unknown status", code
    assert "timed out" in rra.rra_status_string(rra.RRA_ERR_TIMEOUT)
    assert "workspace" in rra.rra_status_string(rra.RRA_ERR_WORKSPACE)
    assert rra.RRA_OK == rra.RRA_SUCCESS == 0


def test_finalize_without_init_is_a_no_op(lib):
    assert rra.rra_finalize() == rra.RRA_OK


@pytest.mark.parametrize("B", [0, 1, 3, 4, 5, 119, 120, 121, 1 << 20])
def test_wire_sizes(lib, B):
    assert rra.rra_ll_wire_bytes(B) == 8 * math.ceil(B / 4)
    assert rra.rra_ll128_wire_bytes(B) == 128 * math.ceil(B / 120)


def _ar(bufs, outs, n, count, dtype=rra.RRA_FLOAT32, op=rra.RRA_SUM, algo=rra.RRA_ALGO_ONE_SHOT):
    return rra.rra_allreduce(bufs, outs, count, dtype, op, algo, check=False, nranks=n)


def test_argument_errors_return_before_launch(lib):
    A = 1 << 40  # fake, never dereferenced: every case fails validation first
    ins = [A + i * (1 << 30) for i in range(8)]
    outs = [A + (16 << 30) + i * (1 << 30) for i in range(8)]
    assert _ar(ins, outs, 0, 10) == rra.RRA_ERR_INVALID_ARG
    assert _ar(ins + [A], outs + [A], 9, 10) == rra.RRA_ERR_UNSUPPORTED
    assert _ar(ins, outs, 2, 10, dtype=7) == rra.RRA_ERR_INVALID_ARG
    assert _ar(ins, outs, 2, 10, op=3) == rra.RRA_ERR_INVALID_ARG
    assert _ar(ins, outs, 2, 10, algo=9) == rra.RRA_ERR_INVALID_ARG
    assert _ar(ins, outs, 2, 10, algo=rra.RRA_ALGO_DIRECT) == rra.RRA_ERR_INVALID_ARG
    assert _ar([0, ins[1]], outs, 2, 10) == rra.RRA_ERR_INVALID_ARG
    assert _ar([ins[0] + 2, ins[1]], outs, 2, 10) == rra.RRA_ERR_INVALID_ARG  # not float-aligned
    # bfloat16 needs only 2-byte alignment
    assert _ar([ins[0] + 2, ins[1]], outs, 2, 0, dtype=rra.RRA_BFLOAT16) == rra.RRA_SUCCESS
    # overlapping outputs, output inside another rank's input
    assert _ar(ins, [outs[0], outs[0] + 8], 2, 10) == rra.RRA_ERR_ALIAS
    assert _ar(ins, [ins[1], outs[1]], 2, 10) == rra.RRA_ERR_ALIAS
    assert _ar(ins, [ins[0] + 4, outs[1]], 2, 10) == rra.RRA_ERR_ALIAS  # partial overlap
    # in place is fine; count 0 launches nothing
    assert _ar(ins, ins, 8, 0) == rra.RRA_SUCCESS
    assert _ar(ins, outs, 8, 0, algo=rra.RRA_ALGO_RING) == rra.RRA_SUCCESS


def test_rs_ag_argument_errors(lib):
    A = 1 << 40
    ins = [A + i * (1 << 30) for i in range(4)]
    outs = [A + (16 << 30) + i * (1 << 30) for i in range(4)]
    rs = lambda o, algo=rra.RRA_ALGO_DIRECT, c=10: rra.rra_reduce_scatter(
        ins, o, c, rra.RRA_FLOAT32, rra.RRA_SUM, algo, check=False, nranks=4)
    ag = lambda b, o, algo=rra.RRA_ALGO_DIRECT, c=10: rra.rra_all_gather(
        b, o, c, rra.RRA_FLOAT32, algo, check=False, nranks=4)
    assert rs(outs, rra.RRA_ALGO_ONE_SHOT) == rra.RRA_ERR_INVALID_ARG
    # in place RS: out r at slice r of its own input
    assert rs([ins[r] + r * 40 for r in range(4)], c=0) == rra.RRA_SUCCESS
    assert rs([ins[r] + 40 for r in range(4)]) == rra.RRA_ERR_ALIAS
    assert ag(ins, outs, rra.RRA_ALGO_ONE_SHOT) == rra.RRA_ERR_INVALID_ARG
    # in place AG: shard r at slot r of its own output
    assert ag([outs[r] + r * 40 for r in range(4)], outs, c=0) == rra.RRA_SUCCESS
    assert ag([outs[r] for r in range(4)], outs) == rra.RRA_ERR_ALIAS


def test_ll_argument_errors(lib):
    A = 1 << 40
    assert rra.rra_ll_pack(A, A + (1 << 30), 0, payload_bytes=16, check=False) == rra.RRA_ERR_INVALID_ARG
    assert rra.rra_ll_pack(A, A + (1 << 30) + 8, 1, payload_bytes=16, check=False) == rra.RRA_ERR_INVALID_ARG
    assert rra.rra_ll128_pack(A, A + 64, 1, payload_bytes=1024, check=False) == rra.RRA_ERR_ALIAS
    wires = [A + i * (1 << 30) for i in range(9)]
    out = A + (32 << 30)
    u = lambda w, **k: rra.rra_ll_unpack(w, out, 1, dtype=rra.RRA_INT32, payload_bytes=k.get("B", 64),
                                          check=False, nsrc=k.get("nsrc", len(w)))
    assert u(wires[:9]) == rra.RRA_ERR_UNSUPPORTED
    assert u(wires[:2], B=6) == rra.RRA_ERR_INVALID_ARG  # not whole int32 elements
    assert rra.rra_ll128_unpack(wires[:2], out, 0, dtype=rra.RRA_INT32, payload_bytes=64,
                                check=False) == rra.RRA_ERR_INVALID_ARG


def test_flight_recorder_records_rejections(lib):
    A = 1 << 40
    rra.rra_allreduce([A, A + (1 << 30)], [A + (2 << 30), A + (3 << 30)], 0, rra.RRA_INT32,
                      rra.RRA_SUM, rra.RRA_ALGO_RING, check=False)
    rra.rra_allreduce([A, A + (1 << 30)], [A + (2 << 30), A + (2 << 30)], 5, rra.RRA_INT32,
                      rra.RRA_SUM, rra.RRA_ALGO_RING, check=False)
    text = rra.rra_dump_recent().strip().splitlines()
    assert "algo=ring n=2 count=0 dtype=int32" in text[-2] and text[-2].endswith("status=success")
    assert text[-1].endswith("status=buffers overlap")


def test_selector_prior_and_tuning_table(lib, tmp_path):
    rra.rra_load_tuning(None)
    # prior: on one GPU one-shot moves the floor bytes with the fewest
    # synchronizations, so it is chosen at every size and rank count
    for n in (1, 2, 3, 5, 8):
        for size in (1, 4096, 1 << 20, 1 << 30):
            assert rra.rra_select_algo(n, size, rra.RRA_BFLOAT16) == rra.RRA_ALGO_ONE_SHOT
    p = tmp_path / "tune.txt"
    p.write_text("# n dtype log2_bytes algo\n8 float32 10 ring\n8 float32 20 two_shot\n"
                 "8 float32 26 one_shot  # big\n4 int32 0 ring\n")
    rra.rra_load_tuning(str(p))
    assert rra.rra_select_algo(8, 1024, rra.RRA_FLOAT32) == rra.RRA_ALGO_RING
    assert rra.rra_select_algo(8, (1 << 20) + 1, rra.RRA_FLOAT32) == rra.RRA_ALGO_TWO_SHOT
    assert rra.rra_select_algo(8, 1 << 30, rra.RRA_FLOAT32) == rra.RRA_ALGO_ONE_SHOT
    assert rra.rra_select_algo(4, 7, rra.RRA_INT32) == rra.RRA_ALGO_RING
    bad = tmp_path / "bad.txt"
    bad.write_text("8 float32 10 warp_drive\n")
    assert rra.rra_load_tuning(str(bad), check=False) == rra.RRA_ERR_INVALID_ARG
    assert rra.rra_select_algo(8, 1024, rra.RRA_FLOAT32) == rra.RRA_ALGO_RING  # old table kept
    rra.rra_load_tuning(None)


def test_fitted_alpha_beta_prior(lib, tmp_path):
    """Where the table has no row for (n, dtype), the fitted alpha-beta
    prior picks the schedule with the least alpha * syncs(n) + beta * n * S
    (syncs: ring 2(n-1), one-shot 1, two-shot 2, tree 2 ceil(log2 n)).
    With one-shot at alpha 1 us, beta 2 us per MiB of n*S and two-shot at
    alpha 4 us (two syncs: 8 us), beta 1 us per MiB, one-shot is faster
    while 1 + 2x < 8 + x, i.e. below x = n*S = 7 MiB."""
    p = tmp_path / "prior.txt"
    p.write_text("ab float32 one_shot 1.0 2.0\nab float32 two_shot 4.0 1.0\n"
                 "ab float32 ring 100.0 1.0\n8 int32 10 ring\n")
    rra.rra_load_tuning(str(p))
    try:
        # n = 4: x = 4 S / MiB; crossover at S = 7/4 MiB
        assert rra.rra_select_algo(4, 1 << 20, rra.RRA_FLOAT32) == rra.RRA_ALGO_ONE_SHOT
        assert rra.rra_select_algo(4, 2 << 20, rra.RRA_FLOAT32) == rra.RRA_ALGO_TWO_SHOT
        # n = 7: crossover at S = 1 MiB
        assert rra.rra_select_algo(7, (1 << 20) - 4096, rra.RRA_FLOAT32) == rra.RRA_ALGO_ONE_SHOT
        assert rra.rra_select_algo(7, (1 << 20) + 4096, rra.RRA_FLOAT32) == rra.RRA_ALGO_TWO_SHOT
        # the table's rows still win for their (n, dtype); other types fall
        # back to one-shot with no prior of their own
        assert rra.rra_select_algo(8, 1 << 10, rra.RRA_INT32) == rra.RRA_ALGO_RING
        assert rra.rra_select_algo(8, 1 << 30, rra.RRA_BFLOAT16) == rra.RRA_ALGO_ONE_SHOT
    finally:
        rra.rra_load_tuning(None)
    bad = tmp_path / "bad_prior.txt"
    bad.write_text("ab float32 one_shot -1 2\n")
    assert rra.rra_load_tuning(str(bad), check=False) == rra.RRA_ERR_INVALID_ARG


def test_shipped_tuning_table(lib):
    # the table made by the size sweep on a GB300 loads, covers n = 2, 4, 8
    # for int32, bfloat16 and float32 from 1 KiB to 1 GiB, and the selector
    # returns its pick at every point; below 64 MiB per rank, where a call
    # is bound by its synchronizations, the pick is one-shot (one sync); the
    # fitted prior picks one-shot for rank counts the table lacks
    path = os.path.join(os.path.dirname(rra.__file__), "tune", "gb300.txt")
    lines = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    rows = [r for r in lines if r[0] != "ab"]
    prior = [r for r in lines if r[0] == "ab"]
    types = ("int32", "bfloat16", "float32")
    code = {"ring": rra.RRA_ALGO_RING, "one_shot": rra.RRA_ALGO_ONE_SHOT, "two_shot": rra.RRA_ALGO_TWO_SHOT,
            "tree": rra.RRA_ALGO_TREE}
    dcode = {"int32": rra.RRA_INT32, "bfloat16": rra.RRA_BFLOAT16, "float32": rra.RRA_FLOAT32}
    assert {(int(r[0]), r[1]) for r in rows} == {(n, d) for n in (2, 4, 8) for d in types}
    assert {int(r[2]) for r in rows} == set(range(10, 31))
    assert {r[3] for r in rows} <= set(code)
    # the fitted prior covers every type and schedule
    assert {(r[1], r[2]) for r in prior} == {(d, a) for d in types for a in ("ring", "one_shot", "two_shot", "tree")}
    assert rra.rra_load_tuning(path) == rra.RRA_SUCCESS
    try:
        for n, dt, lb, algo in rows:
            assert rra.rra_select_algo(int(n), 1 << int(lb), dcode[dt]) == code[algo], (n, dt, lb)
            if int(lb) < 26:
                assert algo == "one_shot", (n, dt, lb)
        for n in (3, 5, 6, 7):
            for size in (1 << 10, 1 << 30):
                assert rra.rra_select_algo(n, size, rra.RRA_FLOAT32) == rra.RRA_ALGO_ONE_SHOT
    finally:
        rra.rra_load_tuning(None)
