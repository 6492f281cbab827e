#!/usr/bin/env python3
"""Benchmark: all-reduce HBM GB/s over N virtual ranks on one GB300.

One step is one pass of the whole hot path over one batch of synthetic
input resident in HBM:

* the gradient bucket: n = 8 virtual ranks, float32, 25,000,000 elements
  (100 MB) per rank, normal(0, 1e-2):
  ring all-reduce, one-shot all-reduce, two-shot all-reduce,
  ring reduce-scatter, direct reduce-scatter (input = the bucket),
  ring all-gather, direct all-gather (input = 3,125,000-element shards);
* the LL / LL128 payloads: 4 sources of 256 MiB int32 in [-2^20, 2^20],
  flag = step counter: 4 packs and one 4-source unpack-reduce per format.

value = floor bytes of the step (every input read once, every output
written once, per operation) / device time of the step, in GB/s.  Inputs
(800 MB per all-reduce, 1 GiB of LL payload) are larger than the 129 MB L2,
so no flush is needed between operations.

--impl reference times the CPU oracle on a bounded sample of the same step.
--sweep FILE writes the message-size sweep (1 KiB .. 1 GiB per rank,
n = 2, 4, 8, int32 and bfloat16, every schedule) as JSON lines and a
tuning table for the selector; with --sweep-cold every timed call follows
a write of twice the L2 size (cold L2), hot L2 otherwise.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "allreduce HBM GB/s (% of 8 TB/s) & busbw vs msg size, N virtual ranks, 1 GB300"
UNIT = "GB/s"
N_RANKS = 8
BUCKET = 25_000_000
LL_SRC = 4
LL_BYTES = 256 << 20
WORKLOAD = ("gradient bucket n=8 fp32 25M/rank (ring, one-shot, two-shot AR; ring+direct RS, AG) "
            "+ LL/LL128 pack + 4-source unpack-reduce of 256 MiB int32")
HBM_NOMINAL = 8000.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def l2_copy_peak(torch):
    """GB/s (read + write bytes) of torch's device copy between two 32 MiB
    buffers, which stay in L2 (larger ones spill past one die's share of
    it): a CUDA graph of 50 copies, best of 10 replays.  The denominator for
    kernels whose bound is L2 traffic rather than HBM."""
    n = (32 << 20) // 4
    a = torch.ones(n, dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(5):
            b.copy_(a)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(50):
            b.copy_(a)
    best = None
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        with torch.cuda.stream(s):
            g.replay()
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 50
        best = ms if best is None or ms < best else best
    return 2 * n * 4 / (best / 1e3) / 1e9


def ring_l2_bytes(n, S):
    """Bytes the L2-link ring moves through L2 per all-reduce of S bytes per
    rank (4-byte types): inputs read once (n S; the first reduce-scatter
    message is the sender's input tile, read by the receiver instead of the
    sender), outputs written once (n S), each of the other n-2
    reduce-scatter partials per rank written to a FIFO slot and read back
    (2 (n-2) S over all ranks), and each of the n-1 forwarded values per rank
    read from the sender's output ((n-1) S)."""
    if n < 2:
        return 2 * n * S
    return 2 * n * S + 2 * (n - 2) * S + (n - 1) * S


# --------------------------------------------------------------------------
# clocks (nvidia-smi sampled during the timed region)
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 7:
                continue
            try:
                sm.append(float(p[0]))
                mx = float(p[1])
            except ValueError:
                continue
            for name, v in zip(names, p[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# the step
# --------------------------------------------------------------------------
def floor_bytes(op, n, S, e=4):
    """Bytes a call must move at least: every input read once, every output
    written once (S = per-rank message bytes as the op defines it)."""
    if op.startswith("ar_"):
        return 2 * n * S
    if op.startswith("rs_"):  # S = per-rank input (n * recvcount elements)
        return n * S + S
    if op.startswith("ag_"):  # S = per-rank output (n * sendcount elements)
        return S + n * S
    raise ValueError(op)


def bus_factor(op, n):
    return 2 * (n - 1) / n if op.startswith("ar_") else (n - 1) / n


# the kernel each bench operation launches (the ring's three operations
# share one)
KERNEL_OF = {"ar_ring": "ring_staged_kernel", "rs_ring": "ring_staged_kernel", "ag_ring": "ring_staged_kernel",
             "ar_oneshot": "oneshot_kernel", "ar_twoshot": "twoshot_kernel", "rs_direct": "direct_rs_kernel",
             "ag_direct": "direct_ag_kernel", "ll_pack": "ll_pack_kernel", "ll_unpack": "ll_unpack_kernel",
             "ll128_pack": "ll128_pack_kernel", "ll128_unpack": "ll128_unpack_kernel"}


def dominant(ops, per_op):
    """The kernel with the largest share of the step's device time, summed
    over the operations that launch it, reported on its longest operation
    (floor bytes and time both cover all of that operation's launches, so
    their ratio is the per-launch rate): (kernel, operation, floor bytes,
    share)."""
    share = {}
    for name, _, _, _ in ops:
        share[KERNEL_OF[name]] = share.get(KERNEL_OF[name], 0.0) + per_op[name]
    kernel = max(share, key=share.get)
    name, fb = max(((o[0], o[1]) for o in ops if KERNEL_OF[o[0]] == kernel), key=lambda o: per_op[o[0]])
    return kernel, name, fb, share[kernel] / sum(per_op[o[0]] for o in ops)


class Step:
    """Device buffers and the sequence of C-ABI calls of one step."""

    def __init__(self, torch, rra, inputs, seed, scale=1):
        self.torch, self.rra = torch, rra
        n = N_RANKS
        self.count = BUCKET // scale
        self.rc = self.count // n
        self.llb = LL_BYTES // scale
        dev = torch.device("cuda", torch.cuda.current_device())
        xs = inputs.cfg_gradient_bucket(self.count, seed=seed)
        shards = [x[: self.rc].copy() for x in xs]
        ps = inputs.cfg_ll_payloads(self.llb, LL_SRC, seed=seed)
        self.host = {"bucket": xs, "shards": shards, "payloads": ps}
        self.x = [torch.from_numpy(x).to(dev) for x in xs]
        self.sh = [torch.from_numpy(x).to(dev) for x in shards]
        self.pl = [torch.from_numpy(p).to(dev) for p in ps]
        self.ar_out = [torch.empty_like(t) for t in self.x]
        self.rs_out = [torch.empty(self.rc, dtype=torch.float32, device=dev) for _ in range(n)]
        self.ag_out = [torch.empty(self.rc * n, dtype=torch.float32, device=dev) for _ in range(n)]
        self.ll_w = [torch.zeros(rra.rra_ll_wire_bytes(self.llb), dtype=torch.uint8, device=dev)
                     for _ in range(LL_SRC)]
        self.l8_w = [torch.zeros(rra.rra_ll128_wire_bytes(self.llb), dtype=torch.uint8, device=dev)
                     for _ in range(LL_SRC)]
        self.ll_out = torch.empty(self.llb // 4, dtype=torch.int32, device=dev)
        self.l8_out = torch.empty(self.llb // 4, dtype=torch.int32, device=dev)
        S = self.count * 4
        LW, L8 = rra.rra_ll_wire_bytes(self.llb), rra.rra_ll128_wire_bytes(self.llb)
        B = self.llb
        # (name, floor bytes, launches, bus bytes for busbw or None)
        self.ops = [
            ("ar_ring", floor_bytes("ar_", n, S), 1, S),
            ("ar_oneshot", floor_bytes("ar_", n, S), 1, S),
            ("ar_twoshot", floor_bytes("ar_", n, S), 1, S),
            ("rs_ring", floor_bytes("rs_", n, S), 1, S),
            ("rs_direct", floor_bytes("rs_", n, S), 1, S),
            ("ag_ring", floor_bytes("ag_", n, S), 1, S),
            ("ag_direct", floor_bytes("ag_", n, S), 1, S),
            ("ll_pack", LL_SRC * (B + LW), LL_SRC, None),
            ("ll_unpack", LL_SRC * LW + B, 1, None),
            ("ll128_pack", LL_SRC * (B + L8), LL_SRC, None),
            ("ll128_unpack", LL_SRC * L8 + B, 1, None),
        ]
        self.flag = 0

    def run_op(self, name, stream):
        rra, n = self.rra, N_RANKS
        F, SUM = rra.RRA_FLOAT32, rra.RRA_SUM
        if name == "ar_ring":
            rra.rra_allreduce(self.x, self.ar_out, self.count, F, SUM, rra.RRA_ALGO_RING, stream)
        elif name == "ar_oneshot":
            rra.rra_allreduce(self.x, self.ar_out, self.count, F, SUM, rra.RRA_ALGO_ONE_SHOT, stream)
        elif name == "ar_twoshot":
            rra.rra_allreduce(self.x, self.ar_out, self.count, F, SUM, rra.RRA_ALGO_TWO_SHOT, stream)
        elif name == "ar_tree":  # a row beyond the step (profiling only)
            rra.rra_allreduce(self.x, self.ar_out, self.count, F, SUM, rra.RRA_ALGO_TREE, stream)
        elif name == "rs_ring":
            rra.rra_reduce_scatter(self.x, self.rs_out, self.rc, F, SUM, rra.RRA_ALGO_RING, stream)
        elif name == "rs_direct":
            rra.rra_reduce_scatter(self.x, self.rs_out, self.rc, F, SUM, rra.RRA_ALGO_DIRECT, stream)
        elif name == "ag_ring":
            rra.rra_all_gather(self.sh, self.ag_out, self.rc, F, rra.RRA_ALGO_RING, stream)
        elif name == "ag_direct":
            rra.rra_all_gather(self.sh, self.ag_out, self.rc, F, rra.RRA_ALGO_DIRECT, stream)
        elif name == "ll_pack":
            for p, w in zip(self.pl, self.ll_w):
                rra.rra_ll_pack(p, w, self.flag, stream=stream)
        elif name == "ll_unpack":
            rra.rra_ll_unpack(self.ll_w, self.ll_out, self.flag, stream=stream)
        elif name == "ll128_pack":
            for p, w in zip(self.pl, self.l8_w):
                rra.rra_ll128_pack(p, w, self.flag, stream=stream)
        elif name == "ll128_unpack":
            rra.rra_ll128_unpack(self.l8_w, self.l8_out, self.flag, stream=stream)
        else:
            raise ValueError(name)

    def launches(self):
        return sum(k for _, _, k, _ in self.ops)

    def floor(self):
        return sum(b for _, b, _, _ in self.ops)


def check_consistency(torch, step, stream):
    """Cross-schedule agreement on the bench's own outputs, without the
    oracle (element-by-element parity with the oracle is what the tests
    check): one-shot and two-shot sum every element in the same ascending
    rank order, so their float32 results agree bit for bit on every rank;
    the direct reduce-scatter's slice r is slice r of that sum; the direct
    and ring all-gathers copy every shard unchanged.  Runs each operation
    once more after the timed region."""
    n, rc = N_RANKS, step.rc
    with torch.cuda.stream(stream):
        step.run_op("ar_oneshot", stream)
    torch.cuda.synchronize()
    one = [t.clone() for t in step.ar_out]
    ok = True
    for name in ("ar_twoshot",):
        with torch.cuda.stream(stream):
            step.run_op(name, stream)
        torch.cuda.synchronize()
        ok = ok and all(torch.equal(one[r], step.ar_out[r]) for r in range(n))
    with torch.cuda.stream(stream):
        step.run_op("rs_direct", stream)
    torch.cuda.synchronize()
    ok = ok and all(torch.equal(step.rs_out[r], one[r][r * rc:(r + 1) * rc]) for r in range(n))
    for name in ("ag_direct", "ag_ring"):
        with torch.cuda.stream(stream):
            step.run_op(name, stream)
        torch.cuda.synchronize()
        ok = ok and all(torch.equal(step.ag_out[r][q * rc:(q + 1) * rc], step.sh[q])
                        for r in range(n) for q in range(n))
    return bool(ok)


def run_ours(args):
    import torch

    import collective_all_reduce_rank_gb300 as rra
    from collective_all_reduce_rank_gb300 import inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    rra.rra_init(local)
    step = Step(torch, rra, inputs, seed=rank)
    stream = torch.cuda.Stream()
    names = [o[0] for o in step.ops]

    def one_step(ev=None):
        step.flag += 1
        for i, name in enumerate(names):
            if ev is not None:
                ev[i][0].record(stream)
            step.run_op(name, stream)
            if ev is not None:
                ev[i][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize()
    st, info = rra.rra_query_status(stream)
    if st != 0:
        raise RuntimeError("device status after warm-up: %d %s" % (st, info))

    # timed region: K steps, per-op events on the launching stream
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in names] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for k in range(args.steps):
                one_step(evs[k])
            t1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    st, info = rra.rra_query_status(stream)
    if st != 0:
        raise RuntimeError("device status after the timed steps: %d %s" % (st, info))
    per_op = {n_: statistics.mean(evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(args.steps))
              for i, n_ in enumerate(names)}

    # end to end through the public API: every step copies its inputs from
    # pinned host memory to the device, runs the step, and copies its results
    # back.  Pipelined as a serving loop would be: two device buffer sets
    # alternate; step k+1's inputs copy in (stream s_in) while step k computes
    # and step k-1's results copy out (stream s_out); every reuse of a buffer
    # set waits for the copies and the step that used it before.
    h_x = [torch.from_numpy(x).pin_memory() for x in step.host["bucket"]]
    h_sh = [torch.from_numpy(x).pin_memory() for x in step.host["shards"]]
    h_pl = [torch.from_numpy(p).pin_memory() for p in step.host["payloads"]]

    # the step's results that come back: rank 0's output of every
    # all-reduce and all-gather (identical on every rank), every rank's
    # reduce-scatter slice (they differ), and both unpacked payloads
    def results(st_):
        return ((("ar", st_.ar_out[0]),) + tuple(("rs%d" % r, st_.rs_out[r]) for r in range(N_RANKS)) +
                (("ag", st_.ag_out[0]), ("ll", st_.ll_out), ("l8", st_.l8_out)))

    h_res = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in results(step)}
    h2d = sum(t.numel() * t.element_size() for t in h_x + h_sh + h_pl)
    d2h = sum(t.numel() * t.element_size() for t in h_res.values())
    sets = [step, Step(torch, rra, inputs, seed=rank)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(nsteps):
        ev_in = [torch.cuda.Event() for _ in range(nsteps)]
        ev_cmp = [torch.cuda.Event() for _ in range(nsteps)]
        ev_out = [torch.cuda.Event() for _ in range(nsteps)]
        for k in range(nsteps):
            st_ = sets[k % 2]
            if k >= 2:
                s_in.wait_event(ev_cmp[k - 2])  # the set's last step has read its inputs
            with torch.cuda.stream(s_in):
                for h, d in zip(h_x + h_sh + h_pl, st_.x + st_.sh + st_.pl):
                    d.copy_(h, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if k >= 2:
                stream.wait_event(ev_out[k - 2])  # the set's last results are copied out
            with torch.cuda.stream(stream):
                st_.flag += 1
                for name in names:
                    st_.run_op(name, stream)
                ev_cmp[k].record(stream)
            s_out.wait_event(ev_cmp[k])
            with torch.cuda.stream(s_out):
                for key, d in results(st_):
                    h_res[key].copy_(d, non_blocking=True)
                ev_out[k].record(s_out)

    # the host link of a shared box stalls now and then (one copy of a step
    # measured 55 ms instead of 9.4; two runs of three stalled once): five
    # runs of the pipeline, the median one reported with all five
    e2e_steps = max(3, min(args.steps, 20))
    e2e_run(2)
    torch.cuda.synchronize()
    e2e_runs = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(s_in)
        e2e_run(e2e_steps)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_runs.append(e0.elapsed_time(e1))
    e2e_ms = statistics.median(e2e_runs)
    st, info = rra.rra_query_status(stream)
    if st != 0:
        raise RuntimeError("device status after the end-to-end steps: %d %s" % (st, info))

    consistent = check_consistency(torch, step, stream)

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dist, "cuda")
    if rank != 0:
        dist.destroy_process_group()
        return
    floor = step.floor()
    value = job_throughput(floor, world, args.steps, ms)
    e2e_value = job_throughput(floor, world, e2e_steps, e2e_ms)
    peak, peak_kind = peaks()
    ops = {}
    for name, fb, _, bus in step.ops:
        t = per_op[name]
        d = {"ms": round(t, 4), "GBps": round(fb / (t / 1e3) / 1e9, 1),
             "pct_hbm_8TBps": round(100 * fb / (t / 1e3) / 1e9 / HBM_NOMINAL, 1),
             "frac_of_measured": round(fb / (t / 1e3) / 1e9 / peak, 3)}
        if bus is not None:
            alg = bus / (t / 1e3) / 1e9
            d["algbw"] = round(alg, 1)
            d["busbw"] = round(alg * bus_factor(name, N_RANKS), 1)
        ops[name] = d
    dom_kernel, dom_name, dom_bytes, dom_share = dominant(step.ops, per_op)
    achieved = dom_bytes / (per_op[dom_name] / 1e3) / 1e9
    traffic = load_traffic(dom_name)
    l2_peak = l2_copy_peak(torch)
    l2_extra = None
    if dom_name == "ar_ring":
        l2b = ring_l2_bytes(N_RANKS, step.count * 4)
        l2_ach = l2b / (per_op[dom_name] / 1e3) / 1e9
        l2_extra = {"bound": "l2", "achieved": round(l2_ach, 1), "peak": round(l2_peak, 1),
                    "peak_kind": "measured here: graph of torch copies of an L2-resident 32 MiB buffer",
                    "unit": "GB/s", "frac": round(l2_ach / l2_peak, 3), "l2_bytes_per_launch": l2b}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32,i32",
        "data": "synthetic (seeded numpy PCG64; normal(0,1e-2) fp32 bucket, int32 in [-2^20,2^20])",
        "config": {"workload": WORKLOAD, "n_virtual_ranks": N_RANKS, "bucket_elems_per_rank": step.count,
                   "ll_payload_bytes": step.llb, "ll_sources": LL_SRC,
                   "l2": "inputs larger than L2 (800 MB per AR op, 1 GiB LL payload); no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "op": dom_name,
                     "share": round(dom_share, 3),
                     "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "traffic": traffic, "l2": l2_extra},
        "ops": ops,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "returned": "rank 0's all-reduce and all-gather outputs (the same on every rank), every rank's "
                            "reduce-scatter slice, both unpacked payloads",
                "runs_ms": [round(x, 2) for x in e2e_runs], "of": "the median of five runs",
                "overlap": "step k+1's inputs copy in and step k-1's results copy out while step k runs"},
        "gpu_launches": step.launches() * args.steps,
        "clocks": clk.summary(),
        "consistency_ok": consistent,
    }
    if not args.no_next:
        line["next_rows"] = next_rows(torch, rra, inputs, step, stream)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_scale or 2)
    if not args.no_small:
        line["tp_latency_us"] = tp_latency(torch, rra, inputs, stream)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def time_op(torch, fn, stream, reps=10):
    """Median milliseconds of fn() on `stream` (CUDA events, after warm-up)."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def next_rows(torch, rra, inputs, step, stream):
    """The rows beyond the step's hot path, each timed on its own: the tree
    all-reduce of the bucket, all-reduce + RMSNorm of the 512-token
    activations, the copy-engine all-gather, and GB/s against the SM budget."""
    n, S = N_RANKS, step.count * 4
    F, SUM = rra.RRA_FLOAT32, rra.RRA_SUM
    out = {}
    ms = time_op(torch, lambda: rra.rra_allreduce(step.x, step.ar_out, step.count, F, SUM, rra.RRA_ALGO_TREE,
                                                 stream), stream)
    out["ar_tree_bucket"] = {"ms": round(ms, 4), "GBps": round(2 * n * S / ms / 1e6, 1),
                             "busbw": round(S / ms / 1e6 * bus_factor("ar_", n), 1)}
    ms = time_op(torch, lambda: rra.rra_all_gather(step.sh, step.ag_out, step.rc, F, rra.RRA_ALGO_COPY_ENGINE,
                                                   stream), stream)
    out["ag_copy_engine_bucket"] = {"ms": round(ms, 4), "GBps": round((n + 1) * S / ms / 1e6, 1)}
    t, h = 512, inputs.TP_HIDDEN
    xs = inputs.cfg_tp_activations(t)
    ins = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
    outs = [torch.empty_like(x) for x in ins]
    gamma = torch.ones(h, dtype=torch.bfloat16, device="cuda")
    # microseconds-long calls: a CUDA graph of many, so the host's launch
    # cost is not timed
    tb = n * t * h * 2
    us, _, _ = time_call(torch, lambda: rra.rra_allreduce_rmsnorm(ins, outs, gamma, h, 1e-6, stream=stream), stream, tb)
    us_ar, _, _ = time_call(torch, lambda: rra.rra_allreduce(ins, outs, t * h, rra.RRA_BFLOAT16, SUM,
                                                            rra.RRA_ALGO_ONE_SHOT, stream), stream, tb)
    out["ar_rmsnorm_tp512"] = {"us": round(us, 2), "one_shot_ar_only_us": round(us_ar, 2),
                               "timing": "CUDA graph of 100 calls"}
    budget = {}
    for ctas in (16, 32, 64, 152, 0):
        rra.rra_set_max_ctas(ctas)
        row = {}
        for name, algo in (("one_shot", rra.RRA_ALGO_ONE_SHOT), ("two_shot", rra.RRA_ALGO_TWO_SHOT)):
            ms = time_op(torch, lambda: rra.rra_allreduce(step.x, step.ar_out, step.count, F, SUM, algo, stream),
                         stream, 5)
            row[name] = round(2 * n * S / ms / 1e6, 1)
        budget["all" if ctas == 0 else str(ctas)] = row
    rra.rra_set_max_ctas(0)
    out["sm_budget_GBps"] = budget
    return out


def max_over_ranks(values, dist, device):
    """Element-wise maximum of `values` over all ranks (the slowest replica
    sets the time); identity without a process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(bytes_per_replica_step, world, steps, ms):
    """Whole-job GB/s: every replica moves the same bytes per step; the time
    is the slowest replica's."""
    return world * bytes_per_replica_step * steps / (ms / 1e3) / 1e9


def load_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or
    None when the kernel's source has changed since it was captured."""
    import hashlib

    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[kernel]
    except Exception:
        return None
    src = os.path.join(ROOT, "collective_all_reduce_rank_gb300", "csrc", d["source"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return d["bytes_per_launch"] if h == d["source_sha"] else None


# --------------------------------------------------------------------------
# the oracle as the CPU baseline / reference arm
# --------------------------------------------------------------------------
def oracle_step(oracle, host, flag):
    xs, sh, ps = host["bucket"], host["shards"], host["payloads"]
    B = ps[0].size * 4
    oracle.allreduce("ring", xs, "float32")
    oracle.allreduce("oneshot", xs, "float32")
    oracle.allreduce("twoshot", xs, "float32")
    oracle.reduce_scatter("ring", xs, "float32")
    oracle.reduce_scatter("direct", xs, "float32")
    oracle.all_gather("ring", sh, "float32")
    oracle.all_gather("direct", sh, "float32")
    w = [oracle.ll_pack(p, flag) for p in ps]
    oracle.ll_unpack(w, B, "int32", flag)
    w = [oracle.ll128_pack(p, flag) for p in ps]
    oracle.ll128_unpack(w, B, "int32", flag)


def sample_sizes(share):
    """Bucket elements per rank and LL payload bytes of a 1/share sample,
    rounded down to whole chunks (a multiple of the rank count) and whole
    16-byte groups."""
    count = max(N_RANKS, BUCKET // share // N_RANKS * N_RANKS)
    return count, max(16, LL_BYTES // share // 16 * 16)


def sample_host(scale, seed=0):
    from collective_all_reduce_rank_gb300 import inputs

    count, llb = sample_sizes(scale)
    xs = inputs.cfg_gradient_bucket(count, seed=seed)
    return {"bucket": xs, "shards": [x[: count // N_RANKS].copy() for x in xs],
            "payloads": inputs.cfg_ll_payloads(llb, LL_SRC, seed=seed)}


def sample_floor(scale):
    n = N_RANKS
    count, B = sample_sizes(scale)
    S = count * 4
    LW, L8 = 8 * ((B + 3) // 4), 128 * ((B + 119) // 120)
    return (3 * floor_bytes("ar_", n, S) + 2 * floor_bytes("rs_", n, S) + 2 * floor_bytes("ag_", n, S)
            + LL_SRC * (B + LW) + LL_SRC * LW + B + LL_SRC * (B + L8) + LL_SRC * L8 + B)


def host_cpu():
    """CPU model and the cores this process may run on (the oracle uses one)."""
    model, arm = None, {}
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":")[0].strip().lower()
            if key in ("model name", "cpu model", "hardware") and ":" in line and model is None:
                model = line.split(":", 1)[1].strip()
            elif key in ("cpu implementer", "cpu part") and ":" in line:
                arm.setdefault(key, line.split(":", 1)[1].strip())
    except OSError:
        pass
    if model is None and arm:  # Arm cores list implementer and part codes only
        model = "arm implementer %s part %s" % (arm.get("cpu implementer"), arm.get("cpu part"))
    try:
        avail = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        avail = os.cpu_count()
    return {"cpu_model": model, "host_cores_available": avail}


def cpu_baseline(scale, min_s=10.0, max_steps=8):
    """The oracle on one core: steps at 1/scale of the workload, repeated
    until about `min_s` seconds of CPU work (at most `max_steps`)."""
    import oracle

    host = sample_host(scale)
    count, llb = sample_sizes(scale)
    steps, t = 0, time.perf_counter()
    while True:
        oracle_step(oracle, host, steps + 1)
        steps += 1
        dt = time.perf_counter() - t
        if dt >= min_s or steps >= max_steps:
            break
    return {"value": round(steps * sample_floor(scale) / dt / 1e9, 3), "unit": UNIT, "cores": 1,
            "kind": "oracle", "seconds": round(dt, 2), **host_cpu(),
            "sample": "%d steps at 1/%d of the workload (bucket %d elems/rank, LL payload %d B), "
                      "single-threaded C oracle" % (steps, scale, count, llb),
            "all_cores": cpu_baseline_all_cores(scale)}


def cpu_baseline_all_cores(scale, min_s=2.0, max_rounds=50):
    """The same oracle on every host core this process may use: T threads,
    each running steps on its own independent 1/T share of the sample
    (every element's reduction is independent, so the shares are separate
    problems of the same shape; the C oracle releases the GIL), repeated
    until about `min_s` seconds of wall time."""
    import threading

    import oracle

    T = max(1, min(16, host_cpu()["host_cores_available"] or 1))
    hosts = [sample_host(scale * T, seed=t) for t in range(T)]
    oracle_step(oracle, sample_host(scale * T * 16, seed=T), 1)  # load and build outside the clock
    errs = []

    def work(h, k):
        try:
            oracle_step(oracle, h, k)
        except Exception as e:  # reported below, not swallowed
            errs.append(e)

    rounds, t = 0, time.perf_counter()
    while not errs:
        threads = [threading.Thread(target=work, args=(h, rounds + 1)) for h in hosts]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        rounds += 1
        dt = time.perf_counter() - t
        if dt >= min_s or rounds >= max_rounds:
            break
    if errs:
        raise errs[0]
    return {"value": round(rounds * T * sample_floor(scale * T) / dt / 1e9, 3), "unit": UNIT, "cores": T,
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": "%d threads x %d steps, each on its own 1/%d of the workload; single-threaded "
                      "C oracle per thread" % (T, rounds, scale * T)}


FULL_STEP_CPU_S = 26.0  # one oracle step at full size on one core, measured


def reference_scale(steps, warmup, budget_s=120.0):
    """Sample fraction (a power of two, at least 1/4) that keeps the whole
    reference run near `budget_s` seconds of CPU work."""
    scale = 4
    while (steps + warmup) * FULL_STEP_CPU_S / scale > budget_s and scale < 1024:
        scale *= 2
    return scale


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    if args.cpu_scale is None:
        args.cpu_scale = reference_scale(args.steps, args.warmup)
    host = sample_host(args.cpu_scale)
    for k in range(args.warmup):
        oracle_step(oracle, host, k + 1)
    t = time.perf_counter()
    for k in range(args.steps):
        oracle_step(oracle, host, k + 1)
    dt = time.perf_counter() - t
    value = sample_floor(args.cpu_scale) * args.steps / dt / 1e9
    sample = ("each step = the whole step at 1/%d of the workload, single-threaded C oracle"
              % args.cpu_scale)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32,i32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "n_virtual_ranks": N_RANKS, "sample_scale": args.cpu_scale},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, **host_cpu()},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# tensor-parallel activations: small-message latency
# --------------------------------------------------------------------------
def tp_latency(torch, rra, inputs, stream, reps=100):
    """The tensor-parallel activations (n = 8, bfloat16 [t, 5120], t in
    {1, 8, 32, 512}): microseconds per all-reduce for every schedule and
    AUTO, from a CUDA graph of `reps` calls (the GPU's own time per call) and
    from single launches between events (what one eager call costs, the
    host's launch included), with algbw and busbw of the graph timing."""
    res = {}
    for t in inputs.TP_TOKENS:
        xs = inputs.cfg_tp_activations(t)
        ins = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
        outs = [torch.empty_like(x) for x in ins]
        S = t * inputs.TP_HIDDEN * 2
        row = {}
        for name, algo in (("ring", rra.RRA_ALGO_RING), ("oneshot", rra.RRA_ALGO_ONE_SHOT),
                           ("twoshot", rra.RRA_ALGO_TWO_SHOT), ("tree", rra.RRA_ALGO_TREE),
                           ("auto", rra.RRA_ALGO_AUTO)):
            call = lambda: rra.rra_allreduce(ins, outs, t * inputs.TP_HIDDEN, rra.RRA_BFLOAT16,
                                             rra.RRA_SUM, algo, stream)
            with torch.cuda.stream(stream):
                for _ in range(5):
                    call()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    call()
            g.replay()
            torch.cuda.synchronize()
            samples = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                with torch.cuda.stream(stream):
                    g.replay()
                b.record(stream)
                torch.cuda.synchronize()
                samples.append(a.elapsed_time(b) * 1e3 / reps)
            us = statistics.median(samples)
            single = []
            for _ in range(20):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record(stream)
                    call()
                    b.record(stream)
                torch.cuda.synchronize()
                single.append(a.elapsed_time(b) * 1e3)
            alg = S / (us / 1e6) / 1e9
            row[name] = {"us": round(us, 2), "single_launch_us": round(statistics.median(single), 2),
                         "algbw": round(alg, 1), "busbw": round(alg * 2 * (N_RANKS - 1) / N_RANKS, 1)}
        res["tokens=%d" % t] = row
    return res


# --------------------------------------------------------------------------
# the ring's link forms against size (the protocol crossover)
# --------------------------------------------------------------------------
def run_ring_forms(args):
    """The ring and the tree all-reduce per size in their default form (the
    one the library picks by size) and forced into the staged form (Simple
    links, whole-CTA messages by bulk copies) and the per-warp LL form: n =
    2, 4, 8, fp32 and bf16, 1 KiB .. 16 MiB per rank, a CUDA graph of 50
    calls per point (hot L2).  The forms of a schedule must agree bit for
    bit (the same order); a point where they do not, or where a wait
    expired, stops the run.  An LL tree whose lines do not fit the
    workspace's LL region has no time (null)."""
    import torch

    import collective_all_reduce_rank_gb300 as rra
    from collective_all_reduce_rank_gb300 import inputs

    torch.cuda.set_device(0)
    rra.rra_init(0)
    stream = torch.cuda.Stream()
    out = open(args.ring_forms, "w")
    for algo, code_algo, env in (("ring", rra.RRA_ALGO_RING, "RRA_RING_PROTO"),
                                 ("tree", rra.RRA_ALGO_TREE, "RRA_TREE_PROTO")):
        for dtype, code in (("float32", rra.RRA_FLOAT32), ("bfloat16", rra.RRA_BFLOAT16)):
            for n in inputs.SWEEP_RANKS:
                for k in range(10, 25):
                    S = 1 << k
                    xs = inputs.cfg_sweep(n, S, dtype, seed=S + n)
                    count = xs[0].size
                    if dtype == "bfloat16":
                        ins = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
                    else:
                        ins = [torch.from_numpy(x).cuda() for x in xs]
                    outs = [torch.empty_like(x) for x in ins]
                    call = lambda: rra.rra_allreduce(ins, outs, count, code, rra.RRA_SUM, code_algo, stream)
                    row = {"algo": algo, "dtype": dtype, "n": n, "bytes_per_rank": S}
                    row["default_us"], _, _ = time_call(torch, call, stream, 0)
                    ref = [o.clone() for o in outs]
                    for form in ("staged", "ll"):
                        os.environ[env] = form
                        try:
                            st = rra.rra_allreduce(ins, outs, count, code, rra.RRA_SUM, code_algo, stream,
                                                   check=False)
                            if st == rra.RRA_ERR_WORKSPACE:
                                row[form + "_us"] = None
                                continue
                            row[form + "_us"], _, _ = time_call(torch, call, stream, 0)
                        finally:
                            os.environ.pop(env)
                        if not all(torch.equal(a, b) for a, b in zip(ref, outs)):
                            raise SystemExit("%s forms disagree at n=%d %s %d (%s)" % (algo, n, dtype, S, form))
                    st, info = rra.rra_query_status(stream)
                    if st != 0:
                        raise SystemExit("device status %d %s" % (st, info))
                    for key in ("default_us", "staged_us", "ll_us"):
                        if row[key] is not None:
                            row[key] = round(row[key], 2)
                    timed = [f for f in ("staged", "ll") if row[f + "_us"] is not None]
                    row["fastest"] = min(timed, key=lambda f: row[f + "_us"])
                    out.write(json.dumps(row) + "\n")
                    out.flush()
                    print(json.dumps(row), flush=True)
                    del ins, outs, ref
    out.close()


# --------------------------------------------------------------------------
# LL / LL128 payload sweep (config 4)
# --------------------------------------------------------------------------
def run_ll_sweep(args):
    """Pack (one source) and 4-source unpack-reduce of int32 payloads of
    1 KiB .. 256 MiB in the LL and LL128 wire formats, flag = step counter:
    floor GB/s (payload read + wire written for a pack; 4 wires read +
    payload written for an unpack) and the fraction of the measured HBM peak
    where the bytes exceed 4x the L2 (hot L2 below that)."""
    import torch

    import collective_all_reduce_rank_gb300 as rra
    from collective_all_reduce_rank_gb300 import inputs

    torch.cuda.set_device(0)
    rra.rra_init(0)
    stream = torch.cuda.Stream()
    peak, _ = peaks()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    out = open(args.ll_sweep, "w")
    flag = 0
    for B in inputs.LL_SIZES:
        ps = [torch.from_numpy(p).cuda() for p in inputs.cfg_ll_payloads(B, LL_SRC, seed=B)]
        res = torch.empty(B // 4, dtype=torch.int32, device="cuda")
        for fmt, wb, pack, unpack in (("ll", rra.rra_ll_wire_bytes(B), rra.rra_ll_pack, rra.rra_ll_unpack),
                                      ("ll128", rra.rra_ll128_wire_bytes(B), rra.rra_ll128_pack,
                                       rra.rra_ll128_unpack)):
            wires = [torch.zeros(wb, dtype=torch.uint8, device="cuda") for _ in range(LL_SRC)]
            flag += 1
            f = flag
            for p, w in zip(ps, wires):
                pack(p, w, f, stream=stream)
            torch.cuda.synchronize()
            us_p, p10p, p90p = time_call(torch, lambda: pack(ps[0], wires[0], f, stream=stream), stream, B + wb)
            us_u, p10u, p90u = time_call(torch, lambda: unpack(wires, res, f, stream=stream), stream,
                                         LL_SRC * wb + B)
            st, info = rra.rra_query_status(stream)
            if st != 0:
                raise SystemExit("device status %d %s at %s %d" % (st, info, fmt, B))
            for op, us, p10, p90, fb in (("pack", us_p, p10p, p90p, B + wb),
                                         ("unpack_reduce", us_u, p10u, p90u, LL_SRC * wb + B)):
                gbs = fb / (us / 1e6) / 1e9
                row = {"format": fmt, "op": op, "payload_bytes": B, "sources": LL_SRC if op != "pack" else 1,
                       "wire_bytes": wb, "us": round(us, 3), "us_p10": round(p10, 3), "us_p90": round(p90, 3),
                       "floor_bytes": fb, "GBps": round(gbs, 1), "frac_of_measured": round(gbs / peak, 3),
                       "l2": "hot" if fb < 4 * l2 else "exceeds 4x L2"}
                out.write(json.dumps(row) + "\n")
                out.flush()
                print(json.dumps(row), flush=True)
        del ps, res
        torch.cuda.empty_cache()
    out.close()


# --------------------------------------------------------------------------
# one-shot / direct reduce-scatter / direct all-gather: resident against
# covering grid
# --------------------------------------------------------------------------
DIRECT_SIZES = tuple(4 << (20 + 2 * k) for k in range(5))  # 4 MiB .. 1 GiB per rank, x4


def run_direct_sweep(args):
    """One-shot all-reduce, direct reduce-scatter and direct all-gather of
    n = 2, 4, 8 ranks x 4 MiB .. 1 GiB per rank (float32, bfloat16; the
    sweep's seeded recipe), each timed with RRA_DIRECT_GRID=resident and
    with the library's default grid choice (covering from its thresholds).
    The two forms' outputs are compared bit for bit at every point (parity
    with the oracle is the tests' job)."""
    import torch

    import collective_all_reduce_rank_gb300 as rra
    from collective_all_reduce_rank_gb300 import inputs

    torch.cuda.set_device(0)
    rra.rra_init(0)
    stream = torch.cuda.Stream()
    peak, _ = peaks()
    out = open(args.direct_sweep, "w")
    codes = {"float32": (rra.RRA_FLOAT32, 4), "bfloat16": (rra.RRA_BFLOAT16, 2)}

    def last_grid():
        return int(rra.rra_dump_recent().strip().splitlines()[-1].split("grid=")[1].split()[0])

    try:
        for dtype, (code, e) in codes.items():
            for n in (2, 4, 8):
                for S in DIRECT_SIZES:
                    count = S // e
                    rc = count // n
                    xs = inputs.cfg_sweep(n, S, dtype, seed=S + n)
                    if dtype == "bfloat16":
                        ins = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
                    else:
                        ins = [torch.from_numpy(x).cuda() for x in xs]
                    del xs
                    ar = [torch.empty_like(t) for t in ins]
                    rs = [torch.empty(rc, dtype=ins[0].dtype, device="cuda") for _ in range(n)]
                    ag = [torch.empty_like(t) for t in ins]
                    ops = (
                        ("one_shot", 2 * n * S,
                         lambda: rra.rra_allreduce(ins, ar, count, code, rra.RRA_SUM, rra.RRA_ALGO_ONE_SHOT, stream),
                         ar),
                        ("rs_direct", (n + 1) * S,
                         lambda: rra.rra_reduce_scatter(ins, rs, rc, code, rra.RRA_SUM, rra.RRA_ALGO_DIRECT, stream),
                         rs),
                        ("ag_direct", (n + 1) * S,
                         lambda: rra.rra_all_gather(rs, ag, rc, code, rra.RRA_ALGO_DIRECT, stream), ag),
                    )
                    for op, fb, call, outs in ops:
                        res = {}
                        for form in ("resident", "default"):
                            if form == "resident":
                                os.environ["RRA_DIRECT_GRID"] = "resident"
                            else:
                                os.environ.pop("RRA_DIRECT_GRID", None)
                            with torch.cuda.stream(stream):
                                call()
                            torch.cuda.synchronize()
                            grid = last_grid()
                            kept = [t.clone() for t in outs]
                            us, p10, p90 = time_call(torch, call, stream, fb)
                            res[form] = (us, p10, p90, grid, kept)
                        same = all(torch.equal(a.view(torch.int16), b.view(torch.int16))
                                   for a, b in zip(res["resident"][4], res["default"][4]))
                        if not same:
                            raise SystemExit("grid forms differ: %s %s n=%d S=%d" % (op, dtype, n, S))
                        st, info = rra.rra_query_status(stream)
                        if st != 0:
                            raise SystemExit("device status %d %s at %s %s n=%d S=%d" % (st, info, op, dtype, n, S))
                        for form in ("resident", "default"):
                            us, p10, p90, grid, _ = res[form]
                            gbs = fb / (us / 1e6) / 1e9
                            row = {"op": op, "form": form, "dtype": dtype, "n": n, "bytes_per_rank": S,
                                   "grid": grid, "us": round(us, 3), "us_p10": round(p10, 3),
                                   "us_p90": round(p90, 3), "floor_bytes": fb, "GBps": round(gbs, 1),
                                   "frac_of_measured": round(gbs / peak, 3)}
                            out.write(json.dumps(row) + "\n")
                            out.flush()
                            print(json.dumps(row), flush=True)
                        del res
                    del ins, ar, rs, ag
                    torch.cuda.empty_cache()
    finally:
        os.environ.pop("RRA_DIRECT_GRID", None)
    out.close()


# --------------------------------------------------------------------------
# message-size sweep (config 5) and the selector table
# --------------------------------------------------------------------------
SWEEP_DTYPES = ("int32", "bfloat16", "float32")


def sync_steps(algo, n):
    """Synchronizations a schedule needs (the alpha count of the pages'
    alpha-beta model): 2(n-1) ring steps, one for one-shot, two for
    two-shot, 2 ceil(log2 n) for a tree."""
    return {"ring": 2 * (n - 1), "one_shot": 1, "two_shot": 2,
            "tree": 2 * max(1, (n - 1).bit_length())}[algo]


def fit_alpha_beta(rows):
    """Per (dtype, schedule): t = alpha * sync_steps(n) + beta * n * S
    fitted over every (n, S) point of the sweep by least squares on the
    relative error (each point weighted by 1 / t, so microsecond and
    millisecond calls count alike).  alpha in microseconds per
    synchronization, beta in microseconds per MiB of n * S."""
    fits = {}
    keys = sorted({(r["dtype"], r["algo"]) for r in rows})
    for dt, al in keys:
        pts = [r for r in rows if r["dtype"] == dt and r["algo"] == al]
        A = np.array([[sync_steps(al, r["n"]) / r["us"], r["n"] * r["bytes_per_rank"] / 2 ** 20 / r["us"]]
                      for r in pts])
        y = np.ones(len(pts))
        coef, *_ = np.linalg.lstsq(A, y, rcond=None)
        alpha, beta = max(0.0, float(coef[0])), max(1e-6, float(coef[1]))
        fits[(dt, al)] = (alpha, beta)
    return fits


def run_sweep(args):
    import torch

    import collective_all_reduce_rank_gb300 as rra
    from collective_all_reduce_rank_gb300 import inputs

    torch.cuda.set_device(0)
    rra.rra_init(0)
    stream = torch.cuda.Stream()
    peak, _ = peaks()
    algos = (("ring", rra.RRA_ALGO_RING), ("one_shot", rra.RRA_ALGO_ONE_SHOT),
             ("two_shot", rra.RRA_ALGO_TWO_SHOT), ("tree", rra.RRA_ALGO_TREE))
    sizes = [s for s in inputs.SWEEP_SIZES if s <= args.sweep_max]
    tune, rows = [], []
    out = open(args.sweep, "w")
    # cold-L2 mode: a scratch buffer of twice the L2 size is rewritten
    # before every timed call
    l2_bytes = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device="cuda") if args.sweep_cold else None
    codes = {"int32": rra.RRA_INT32, "bfloat16": rra.RRA_BFLOAT16, "float32": rra.RRA_FLOAT32}
    for n in inputs.SWEEP_RANKS:
        for dtype in SWEEP_DTYPES:
            code = codes[dtype]
            for S in sizes:
                # the seeded numpy recipe of the sweep (the tests check the
                # largest size per rank count and type against the oracle)
                xs = inputs.cfg_sweep(n, S, dtype, seed=S + n)
                count = xs[0].size
                if dtype == "bfloat16":
                    ins = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
                else:
                    ins = [torch.from_numpy(x).cuda() for x in xs]
                del xs
                outs = [torch.empty_like(x) for x in ins]
                best, results = None, {}
                for name, algo in algos:
                    call = lambda: rra.rra_allreduce(ins, outs, count, code, rra.RRA_SUM, algo, stream)
                    if flush is None:
                        us, p10, p90 = time_call(torch, call, stream, S * n)
                    else:
                        us, p10, p90 = time_call_cold(torch, call, stream, flush, S * n)
                    st, info = rra.rra_query_status(stream)
                    if st != 0:
                        raise SystemExit("device status %d %s at n=%d %s %d %s" % (st, info, n, dtype, S, name))
                    results[name] = [o.clone() for o in outs] if S * n <= (1 << 30) else [outs[0].clone()]
                    fb = 2 * n * S
                    alg = S / (us / 1e6) / 1e9
                    row = {"n": n, "dtype": dtype, "bytes_per_rank": S, "algo": name, "us": round(us, 3),
                           "us_p10": round(p10, 3), "us_p90": round(p90, 3),
                           "algbw": round(alg, 2), "busbw": round(alg * 2 * (n - 1) / n, 2),
                           "floor_bytes": fb, "GBps": round(fb / (us / 1e6) / 1e9, 1),
                           "pct_hbm_8TBps": round(100 * fb / (us / 1e6) / 1e9 / HBM_NOMINAL, 1),
                           "frac_of_measured": round(fb / (us / 1e6) / 1e9 / peak, 3),
                           "l2_resident": 2 * n * S < 4 * l2_bytes, "l2": "cold" if flush is not None else "hot"}
                    rows.append(row)
                    if best is None or us < best[1]:
                        best = (name, us)
                # consistency without the oracle: int32 sums are exact, so
                # every schedule agrees bit for bit; one-shot and two-shot
                # share the ascending order in every type
                same = lambda a, b: all(torch.equal(x, y) for x, y in zip(a, b))
                ok = same(results["one_shot"], results["two_shot"])
                if dtype == "int32":
                    ok = ok and all(same(results["one_shot"], results[k]) for k in results)
                for row in rows[-len(algos):]:
                    row["consistent"] = bool(ok)
                    out.write(json.dumps(row) + "\n")
                out.flush()
                tune.append((n, dtype, (S - 1).bit_length(), best[0]))
                del ins, outs, results
                torch.cuda.empty_cache()
    out.close()
    fits = fit_alpha_beta(rows)
    with open(args.sweep + ".tune.txt", "w") as f:
        f.write("# nranks dtype log2_bytes algo  (fastest measured schedule per size)\n")
        for n, dtype, lb, name in tune:
            f.write("%d %s %d %s\n" % (n, dtype, lb, name))
        f.write("# ab dtype algo alpha_us_per_sync beta_us_per_MiB_of_nS  (fitted over the sweep)\n")
        for (dt, al), (alpha, beta) in sorted(fits.items()):
            f.write("ab %s %s %.4f %.6f\n" % (dt, al, alpha, beta))


def spread(samples):
    """(median, p10, p90) of a list of timings."""
    q = sorted(samples)
    pick = lambda f: q[min(len(q) - 1, max(0, int(round(f * (len(q) - 1)))))]
    return statistics.median(q), pick(0.1), pick(0.9)


def time_call_cold(torch, call, stream, flush, total_bytes):
    """(median, p10, p90) microseconds of single calls, each after a write
    of `flush` (twice the L2 size) that evicts the call's inputs and the
    previous call's outputs from L2; the flush is outside the events."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    reps = 20 if total_bytes < (2 << 30) else 5
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for k, (a, b) in enumerate(evs):
            flush.fill_(k & 0xFF)
            a.record(stream)
            call()
            b.record(stream)
    torch.cuda.synchronize()
    return spread([a.elapsed_time(b) * 1e3 for a, b in evs])


def time_call(torch, call, stream, total_bytes):
    """Median microseconds per call: a CUDA graph of many calls for small
    messages, runs of back-to-back launches between events for large ones."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    torch.cuda.synchronize()
    if total_bytes < (64 << 20):
        reps = 100
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                call()
        samples = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            with torch.cuda.stream(stream):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            samples.append(a.elapsed_time(b) * 1e3 / reps)
        return spread(samples)
    # large messages: R calls back to back between two events (the host
    # queues launches far faster than these calls run, so no launch gap is
    # timed), median of 5 such runs
    reps = 10 if total_bytes < (2 << 30) else 4
    samples = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                call()
            b.record(stream)
        torch.cuda.synchronize()
        samples.append(a.elapsed_time(b) * 1e3 / reps)
    return spread(samples)


def run_profile(args):
    """Run the listed operations once each on a 1/scale workload (the small
    case the ncu captures use); exits non-zero on a device error."""
    import torch

    import collective_all_reduce_rank_gb300 as rra
    from collective_all_reduce_rank_gb300 import inputs

    torch.cuda.set_device(0)
    rra.rra_init(0)
    step = Step(torch, rra, inputs, seed=0, scale=args.scale)
    stream = torch.cuda.Stream()
    names = [o[0] for o in step.ops] if args.profile == "all" else args.profile.split(",")
    step.flag = 1
    extra = {}
    if "ar_ring_bf16" in names:
        # bfloat16 ring on as many bytes per rank as the float32 bucket
        xs = inputs.make_ranks(N_RANKS, 2 * step.count, "bfloat16", "normal", seed=5)
        extra["bf16_in"] = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
        extra["bf16_out"] = [torch.empty_like(t) for t in extra["bf16_in"]]
    if "ar_twoshot_n2" in names or "ar_oneshot_n2" in names:
        # two ranks of 64 MiB fp32 (256 MiB in and out: past L2)
        xs = inputs.make_ranks(2, (64 << 20) // 4, "float32", "normal", seed=7)
        extra["n2_in"] = [torch.from_numpy(x).cuda() for x in xs]
        extra["n2_out"] = [torch.empty_like(t) for t in extra["n2_in"]]
    if "ar_rmsnorm" in names:
        # tensor-parallel activations [rows, 5120] bfloat16, rows so that the
        # 8 ranks' inputs exceed L2
        rows = 4096
        xs = inputs.make_ranks(N_RANKS, rows * inputs.TP_HIDDEN, "bfloat16", "normal", seed=6)
        extra["tp_in"] = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
        extra["tp_out"] = [torch.empty_like(t) for t in extra["tp_in"]]
        extra["gamma"] = torch.ones(inputs.TP_HIDDEN, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        for name in names:
            if name == "ll_unpack" and "ll_pack" not in names:
                step.run_op("ll_pack", stream)
            if name == "ll128_unpack" and "ll128_pack" not in names:
                step.run_op("ll128_pack", stream)
            if name == "ar_ring_bf16":
                rra.rra_allreduce(extra["bf16_in"], extra["bf16_out"], 2 * step.count, rra.RRA_BFLOAT16,
                                  rra.RRA_SUM, rra.RRA_ALGO_RING, stream)
            elif name in ("ar_twoshot_n2", "ar_oneshot_n2"):
                algo = rra.RRA_ALGO_TWO_SHOT if name == "ar_twoshot_n2" else rra.RRA_ALGO_ONE_SHOT
                rra.rra_allreduce(extra["n2_in"], extra["n2_out"], extra["n2_in"][0].numel(), rra.RRA_FLOAT32,
                                  rra.RRA_SUM, algo, stream)
            elif name == "ar_rmsnorm":
                rra.rra_allreduce_rmsnorm(extra["tp_in"], extra["tp_out"], extra["gamma"], inputs.TP_HIDDEN,
                                          1e-6, stream=stream)
            else:
                step.run_op(name, stream)
    torch.cuda.synchronize()
    st, info = rra.rra_query_status(stream)
    if st != 0:
        raise SystemExit("device status %d %s" % (st, info))
    print(json.dumps({"profile": names, "scale": args.scale, "bucket_elems_per_rank": step.count,
                      "ll_payload_bytes": step.llb}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-scale", type=int, default=None,
                    help="oracle sample = 1/scale of the workload (default: 2 for the CPU baseline, "
                         "sized to the step count for --impl reference)")
    ap.add_argument("--profile", default=None, help="run these ops once (comma list or 'all') and exit")
    ap.add_argument("--scale", type=int, default=4, help="workload fraction for --profile")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the rows beyond the step (tree, RMSNorm, ...)")
    ap.add_argument("--no-small", action="store_true", help="skip the TP-activation latency table")
    ap.add_argument("--ring-forms", default=None,
                    help="write the ring and tree default, staged and LL forms against size to this JSONL file")
    ap.add_argument("--ll-sweep", default=None,
                    help="write the LL / LL128 payload sweep (1 KiB .. 256 MiB, 4 sources) to this JSONL file")
    ap.add_argument("--sweep", default=None, help="write the message-size sweep to this JSONL file")
    ap.add_argument("--direct-sweep", default=None,
                    help="write one-shot / direct RS / direct AG on resident and default grids to this JSONL file")
    ap.add_argument("--sweep-max", type=int, default=1 << 30)
    ap.add_argument("--sweep-cold", action="store_true",
                    help="flush L2 (write twice its size) before every timed call of the sweep")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.profile:
        run_profile(args)
    elif args.sweep:
        run_sweep(args)
    elif args.ll_sweep:
        run_ll_sweep(args)
    elif args.direct_sweep:
        run_direct_sweep(args)
    elif args.ring_forms:
        run_ring_forms(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
