"""The benchmark's multi-replica path on CPU: two gloo ranks, each a replica
with its own time; the job takes the slowest rank's time and every rank's
bytes."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 100.0 - rank]  # rank 1 is slower in the first slot
    got = bench.max_over_ranks(mine, dist, "cpu")
    q.put((rank, got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 100.0]


def test_job_throughput_counts_every_replica():
    import bench

    # 2 replicas x 1 GB per step x 10 steps in 1 s -> 20 GB/s
    assert bench.job_throughput(1e9, 2, 10, 1000.0) == pytest.approx(20.0)
    assert bench.max_over_ranks([1.0, 2.0], None, "cpu") == [1.0, 2.0]


def test_floor_bytes_and_bus_factors():
    import bench
    from oracle import model

    S = 100
    assert bench.floor_bytes("ar_ring", 8, S) == 1600
    assert bench.floor_bytes("rs_direct", 8, S) == 900
    assert bench.floor_bytes("ag_ring", 8, S) == 900
    # the bench's bus factors are the page's (pinned in the oracle tests)
    assert bench.bus_factor("ar_x", 8) == model.bus_factor("allreduce", 8)
    assert bench.bus_factor("rs_x", 8) == model.bus_factor("reducescatter", 8)
    assert bench.bus_factor("ag_x", 8) == model.bus_factor("allgather", 8)
    # the ring's L2 bytes: inputs and outputs once, each reduce-scatter send
    # after the first through a slot (written, read back; the first is the
    # sender's input, read once as part of the inputs), each forwarded value
    # read once from the sender's output -- 35 S at n = 8 for 4-byte types
    assert bench.ring_l2_bytes(8, S) == 35 * S
    assert bench.ring_l2_bytes(2, S) == 5 * S
    assert bench.ring_l2_bytes(1, S) == 2 * S
    # pinned to the oracle's byte counters of an actual ring all-reduce: its
    # reduce-scatter half sends n-1 partials per rank (the first of them the
    # rank's own input), the rest are forwarded values
    import numpy as np
    import oracle

    n = 8
    xs = [np.full(800, k, dtype=np.int32) for k in range(n)]
    _, sent, _ = oracle.allreduce("ring", xs, "int32")
    _, sent_rs, _ = oracle.reduce_scatter("ring", xs, "int32")
    rs, values = int(np.sum(sent_rs)), int(np.sum(sent)) - int(np.sum(sent_rs))
    assert rs == values == 7 * 800 * 4
    slot_partials = rs * (n - 2) // (n - 1)
    assert bench.ring_l2_bytes(n, 800 * 4) == 2 * n * 800 * 4 + 2 * slot_partials + values


def test_cpu_baseline_samples():
    import bench

    # samples are whole chunks and whole 16-byte LL groups at any share
    for share in (1, 2, 3, 7, 24, 64, 1 << 20):
        count, llb = bench.sample_sizes(share)
        assert count % bench.N_RANKS == 0 and count >= bench.N_RANKS
        assert llb % 16 == 0 and llb >= 16
    assert bench.sample_sizes(1) == (bench.BUCKET, bench.LL_BYTES)
    # T independent shares carry the sample's floor bytes, up to the rounding
    full = bench.sample_floor(2)
    for T in (3, 8, 16):
        assert abs(T * bench.sample_floor(2 * T) - full) / full < 1e-4
    # the all-cores variant runs the oracle on every share and reports its threads
    r = bench.cpu_baseline_all_cores(4096, min_s=0.0, max_rounds=1)
    assert r["kind"] == "oracle" and r["cores"] >= 1 and r["value"] > 0


def test_every_bench_op_names_its_kernel():
    # the roofline's dominant kernel is chosen by summed share over the
    # operations that launch it
    import bench

    names = ["ar_ring", "ar_oneshot", "ar_twoshot", "rs_ring", "rs_direct", "ag_ring", "ag_direct", "ll_pack",
             "ll_unpack", "ll128_pack", "ll128_unpack"]
    assert set(names) == set(bench.KERNEL_OF)
    assert {bench.KERNEL_OF[k] for k in ("ar_ring", "rs_ring", "ag_ring")} == {"ring_staged_kernel"}


def test_dominant_kernel_sums_its_operations():
    import bench

    ops = [("ar_ring", 160, 1, 1), ("rs_ring", 90, 1, 1), ("ag_ring", 90, 1, 1), ("ll_unpack", 60, 1, None),
           ("ll_pack", 100, 4, None)]
    # ll_unpack is the longest single operation, but the ring's three add up
    t = {"ar_ring": 0.36, "rs_ring": 0.21, "ag_ring": 0.18, "ll_unpack": 0.37, "ll_pack": 0.50}
    kernel, name, fb, share = bench.dominant(ops, t)
    assert (kernel, name, fb) == ("ring_staged_kernel", "ar_ring", 160)
    assert abs(share - 0.75 / 1.62) < 1e-12
    # a kernel launched four times by one operation can dominate too
    t.update(ll_pack=2.0)
    assert bench.dominant(ops, t)[:3] == ("ll_pack_kernel", "ll_pack", 100)


def test_traffic_capture_matches_the_kernel_source():
    # the bench line's DRAM traffic comes from a committed ncu capture; it
    # must have been taken on the kernel source as it stands (bench.py
    # reports null otherwise)
    import bench

    t = bench.load_traffic("ar_ring")
    assert t is not None and t > 0
