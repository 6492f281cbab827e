"""CPU oracle for the virtual-rank collectives (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never loads it and shares
no code with it.  The arithmetic lives in ``rra_oracle.c`` (plain C, built
with gcc ``-O2 -ffp-contract=off``, no fast-math); this module only compiles
that file on demand and marshals numpy arrays through ctypes.  The alpha-beta
cost model and the bandwidth metrics are in ``oracle.model``.

Data types are named ``"int32"``, ``"float32"`` and ``"bfloat16"``.  Arrays
are numpy ``int32`` / ``float32`` / ``uint16`` (the raw bfloat16 bits).

Parity status: every function here is pinned by ``tests/test_oracle.py``
(closed forms, brute force, the pages' printed values, library routines).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rra_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"int32": 0, "float32": 1, "bfloat16": 2}
NP_DTYPES = {"int32": np.int32, "float32": np.float32, "bfloat16": np.uint16}
ELEM_SIZE = {"int32": 4, "float32": 4, "bfloat16": 2}


def build(force: bool = False) -> str:
    """Compile rra_oracle.c into liboracle.so next to it; return the path."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + ".%d.tmp" % os.getpid()
            cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                   "-Wall", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.check_call(cmd)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    vpp = ctypes.POINTER(ctypes.c_void_p)
    u64p = ctypes.POINTER(ctypes.c_uint64)
    szp = ctypes.POINTER(ctypes.c_size_t)
    for name in ("orc_allreduce_ring", "orc_allreduce_oneshot", "orc_allreduce_twoshot", "orc_allreduce_tree",
                 "orc_reduce_scatter_ring", "orc_reduce_scatter_direct",
                 "orc_all_gather_ring", "orc_all_gather_direct"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_int, vpp, vpp, u64p, u64p]
    lib.orc_chunk_plan.restype = ctypes.c_int
    lib.orc_chunk_plan.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_int, szp]
    lib.orc_ll_wire_bytes.restype = ctypes.c_size_t
    lib.orc_ll_wire_bytes.argtypes = [ctypes.c_size_t]
    lib.orc_ll128_wire_bytes.restype = ctypes.c_size_t
    lib.orc_ll128_wire_bytes.argtypes = [ctypes.c_size_t]
    lib.orc_ll_pack.restype = None
    lib.orc_ll_pack.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint32]
    lib.orc_ll128_pack.restype = None
    lib.orc_ll128_pack.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint64]
    lib.orc_ll_unpack.restype = ctypes.c_longlong
    lib.orc_ll_unpack.argtypes = [vpp, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                  ctypes.c_uint32]
    lib.orc_ll128_unpack.restype = ctypes.c_longlong
    lib.orc_ll128_unpack.argtypes = [vpp, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.c_int, ctypes.c_uint64]
    lib.orc_allreduce_rmsnorm.restype = ctypes.c_int
    lib.orc_allreduce_rmsnorm.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int,
                                          vpp, ctypes.c_void_p, ctypes.c_double, vpp]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.orc_bf16_to_f32.restype = ctypes.c_float
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    _lib = lib
    return lib


def _ptrs(arrays):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def _check(xs, dtype):
    want = NP_DTYPES[dtype]
    for x in xs:
        if x.dtype != want or not x.flags["C_CONTIGUOUS"]:
            raise TypeError("oracle wants C-contiguous %s arrays for %s" % (np.dtype(want), dtype))


def chunk_plan(n: int, count: int, dtype: str) -> list[int]:
    """Chunk edges (n+1 entries) of the ring / two-shot chunk plan."""
    b = (ctypes.c_size_t * (n + 1))()
    if _load().orc_chunk_plan(n, count, DTYPES[dtype], b) != 0:
        raise ValueError("bad chunk plan arguments")
    return list(b)


def _run(fname, xs, out_count, dtype):
    _check(xs, dtype)
    n = len(xs)
    outs = [np.zeros(out_count, dtype=NP_DTYPES[dtype]) for _ in range(n)]
    sent = (ctypes.c_uint64 * n)()
    recv = (ctypes.c_uint64 * n)()
    return outs, sent, recv, _ptrs(xs), _ptrs(outs)


def allreduce(algo: str, xs, dtype: str):
    """All-reduce (SUM) of the n arrays in ``xs`` with schedule ``algo``
    ("ring", "oneshot", "twoshot", "tree").  Returns (outs, sent, recv) where sent and
    recv are per-rank byte counters."""
    count = int(xs[0].size)
    outs, sent, recv, pin, pout = _run(None, xs, count, dtype)
    fn = {"ring": "orc_allreduce_ring", "oneshot": "orc_allreduce_oneshot",
          "twoshot": "orc_allreduce_twoshot", "tree": "orc_allreduce_tree"}[algo]
    rc = getattr(_load(), fn)(len(xs), count, DTYPES[dtype], pin, pout, sent, recv)
    if rc != 0:
        raise RuntimeError("oracle %s failed: %d" % (fn, rc))
    return outs, list(sent), list(recv)


def reduce_scatter(algo: str, xs, dtype: str):
    """Reduce-scatter: xs[r] holds n*rc elements; returns (outs[rc], sent, recv)."""
    n = len(xs)
    if xs[0].size % n:
        raise ValueError("reduce_scatter input must hold n * recvcount elements")
    rc_ = int(xs[0].size // n)
    outs, sent, recv, pin, pout = _run(None, xs, rc_, dtype)
    fn = {"ring": "orc_reduce_scatter_ring", "direct": "orc_reduce_scatter_direct"}[algo]
    rc = getattr(_load(), fn)(n, rc_, DTYPES[dtype], pin, pout, sent, recv)
    if rc != 0:
        raise RuntimeError("oracle %s failed: %d" % (fn, rc))
    return outs, list(sent), list(recv)


def all_gather(algo: str, xs, dtype: str):
    """All-gather: xs[r] holds sc elements; returns (outs[n*sc], sent, recv)."""
    n = len(xs)
    sc = int(xs[0].size)
    outs, sent, recv, pin, pout = _run(None, xs, n * sc, dtype)
    fn = {"ring": "orc_all_gather_ring", "direct": "orc_all_gather_direct"}[algo]
    rc = getattr(_load(), fn)(n, sc, DTYPES[dtype], pin, pout, sent, recv)
    if rc != 0:
        raise RuntimeError("oracle %s failed: %d" % (fn, rc))
    return outs, list(sent), list(recv)


def allreduce_rmsnorm(xs, gamma, eps: float, dtype: str, hidden: int):
    """Fused all-reduce + RMSNorm of rows of `hidden` elements: every rank
    gets RMSNorm(sum_k xs[k]) * gamma.  Returns the n outputs."""
    _check(list(xs) + [gamma], dtype)
    n = len(xs)
    rows = xs[0].size // hidden
    outs = [np.zeros(xs[0].size, dtype=NP_DTYPES[dtype]) for _ in range(n)]
    rc = _load().orc_allreduce_rmsnorm(n, rows, hidden, DTYPES[dtype], _ptrs(xs), gamma.ctypes.data,
                                       eps, _ptrs(outs))
    if rc != 0:
        raise RuntimeError("oracle allreduce_rmsnorm failed: %d" % rc)
    return outs


def ll_wire_bytes(payload_bytes: int) -> int:
    return int(_load().orc_ll_wire_bytes(payload_bytes))


def ll128_wire_bytes(payload_bytes: int) -> int:
    return int(_load().orc_ll128_wire_bytes(payload_bytes))


def ll_pack(payload: np.ndarray, flag: int) -> np.ndarray:
    """Pack the payload's bytes into LL lines; returns the wire as uint8."""
    p = np.ascontiguousarray(payload).view(np.uint8).reshape(-1)
    wire = np.empty(ll_wire_bytes(p.size), dtype=np.uint8)
    _load().orc_ll_pack(p.ctypes.data, p.size, wire.ctypes.data, flag)
    return wire


def ll128_pack(payload: np.ndarray, flag: int) -> np.ndarray:
    p = np.ascontiguousarray(payload).view(np.uint8).reshape(-1)
    wire = np.empty(ll128_wire_bytes(p.size), dtype=np.uint8)
    _load().orc_ll128_pack(p.ctypes.data, p.size, wire.ctypes.data, flag)
    return wire


def _unpack(fn, wires, payload_bytes, dtype, expected):
    out = np.zeros(payload_bytes // ELEM_SIZE[dtype], dtype=NP_DTYPES[dtype])
    ws = [np.ascontiguousarray(w).view(np.uint8) for w in wires]
    bad = getattr(_load(), fn)(_ptrs(ws), len(ws), out.ctypes.data, payload_bytes,
                               DTYPES[dtype], expected)
    if bad == -2:
        raise ValueError("payload size is not a whole number of elements")
    return out, int(bad)


def ll_unpack(wires, payload_bytes: int, dtype: str, expected_flag: int):
    """Unpack-and-reduce LL wires; returns (out, first_bad_line or -1)."""
    return _unpack("orc_ll_unpack", wires, payload_bytes, dtype, expected_flag)


def ll128_unpack(wires, payload_bytes: int, dtype: str, expected_flag: int):
    return _unpack("orc_ll128_unpack", wires, payload_bytes, dtype, expected_flag)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 bits (nearest, ties to even)."""
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in flat], dtype=np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(h, dtype=np.uint16).reshape(-1)
    return np.array([lib.orc_bf16_to_f32(int(v)) for v in flat], dtype=np.float32)
