"""GB300-native all-reduce, reduce-scatter and all-gather over N virtual ranks.

A thin ctypes binding over ``librra.so`` (the C ABI declared in
``include/rra.h``).  Every function here has the C function's name and only
marshals arguments: torch tensors become device pointers, torch streams
become ``cudaStream_t``.  All computation runs in the library's CUDA kernels;
there is no CPU path.  A call whose status is not ``RRA_SUCCESS`` raises
``RraError`` (pass ``check=False`` to get the status code instead).

The library is built in-tree (``collective_all_reduce_rank_gb300/librra.so``)
by ``build.build()``; loading it builds it first when the sources are newer,
and raises if that is impossible.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

RRA_OK = 0
RRA_SUCCESS = RRA_OK
RRA_ERR_INVALID_ARG = 1
RRA_ERR_UNSUPPORTED = 2
RRA_ERR_ALIAS = 3
RRA_ERR_NOT_INITIALIZED = 4
RRA_ERR_CUDA = 5
RRA_ERR_TIMEOUT = 6
RRA_ERR_WORKSPACE = 7

RRA_INT32 = 0
RRA_FLOAT32 = 1
RRA_BFLOAT16 = 2

RRA_SUM = 0

RRA_ALGO_AUTO = 0
RRA_ALGO_RING = 1
RRA_ALGO_ONE_SHOT = 2
RRA_ALGO_TWO_SHOT = 3
RRA_ALGO_DIRECT = 4
RRA_ALGO_COPY_ENGINE = 5
RRA_ALGO_TREE = 6

RRA_MAX_RANKS = 8

DTYPE_NAMES = {RRA_INT32: "int32", RRA_FLOAT32: "float32", RRA_BFLOAT16: "bfloat16"}
ALGO_NAMES = {RRA_ALGO_AUTO: "auto", RRA_ALGO_RING: "ring", RRA_ALGO_ONE_SHOT: "one_shot",
              RRA_ALGO_TWO_SHOT: "two_shot", RRA_ALGO_DIRECT: "direct"}

_lock = threading.Lock()
_lib = None


class RraError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what or "rra", rra_status_string(status), status))


def library_path() -> str:
    return _build.LIB


def load():
    """Load librra.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError("librra.so is missing and could not be built")
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib = lib
    return _lib


def _declare(lib):
    vp = ctypes.c_void_p
    vpp = ctypes.POINTER(ctypes.c_void_p)
    i, sz, u32, u64 = ctypes.c_int, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64
    sigs = {
        "rra_init": (i, [i, sz]),
        "rra_finalize": (i, []),
        "rra_allreduce": (i, [vpp, vpp, i, sz, i, i, i, vp]),
        "rra_allreduce_two_shot_static": (i, [vpp, vpp, i, sz, i, i, vp]),
        "rra_reduce_scatter": (i, [vpp, vpp, i, sz, i, i, i, vp]),
        "rra_all_gather": (i, [vpp, vpp, i, sz, i, i, vp]),
        "rra_allreduce_rmsnorm": (i, [vpp, vpp, i, sz, sz, vp, ctypes.c_float, i, vp]),
        "rra_ll_wire_bytes": (sz, [sz]),
        "rra_ll128_wire_bytes": (sz, [sz]),
        "rra_ll_pack": (i, [vp, sz, vp, u32, vp]),
        "rra_ll_unpack": (i, [vpp, i, vp, sz, i, i, u32, vp]),
        "rra_ll128_pack": (i, [vp, sz, vp, u64, vp]),
        "rra_ll128_unpack": (i, [vpp, i, vp, sz, i, i, u64, vp]),
        "rra_query_status": (i, [vp, ctypes.POINTER(ctypes.c_int32)]),
        "rra_query_status_static": (i, [vp, ctypes.POINTER(ctypes.c_int32)]),
        "rra_select_algo": (i, [i, sz, i]),
        "rra_load_tuning": (i, [ctypes.c_char_p]),
        "rra_set_timeout_ns": (None, [u64]),
        "rra_debug_skip_rank": (None, [i]),
        "rra_set_max_ctas": (None, [i]),
        "rra_status_string": (ctypes.c_char_p, [i]),
        "rra_dump_recent": (i, [ctypes.c_char_p, sz]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def header_symbols() -> list[str]:
    """Names of every function include/rra.h declares."""
    hdr = os.path.join(_build.ROOT, "include", "rra.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rra_[a-z0-9_]+)\s*\(", text)))


# ---------------------------------------------------------------------------
# marshalling
# ---------------------------------------------------------------------------

def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("tensors passed to rra must be contiguous")
        return int(x.data_ptr())
    raise TypeError("expected a tensor or a device pointer (int), got %r" % type(x))


def _ptr_array(xs):
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _stream(stream, like=None) -> int:
    if stream is None:
        if like is not None and hasattr(like, "device"):
            import torch

            return int(torch.cuda.current_stream(like.device).cuda_stream)
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _dtype_of(t):
    import torch

    m = {torch.int32: RRA_INT32, torch.float32: RRA_FLOAT32, torch.bfloat16: RRA_BFLOAT16}
    if t.dtype not in m:
        raise TypeError("unsupported dtype %s (int32, float32, bfloat16)" % t.dtype)
    return m[t.dtype]


def _resolve(xs, count, dtype):
    first = xs[0] if xs else None
    if dtype is None:
        if first is None or isinstance(first, int):
            raise ValueError("dtype is required with raw pointers")
        dtype = _dtype_of(first)
    if count is None:
        if first is None or isinstance(first, int):
            raise ValueError("count is required with raw pointers")
        count = int(first.numel())
    return count, dtype


def _ret(status, what, check):
    if check and status != RRA_SUCCESS:
        raise RraError(status, what)
    return status


# ---------------------------------------------------------------------------
# the C functions
# ---------------------------------------------------------------------------

def rra_status_string(status: int) -> str:
    return load().rra_status_string(status).decode()


def rra_init(device: int = 0, workspace_bytes: int = 0, check: bool = True) -> int:
    return _ret(load().rra_init(device, workspace_bytes), "rra_init", check)


def rra_finalize(check: bool = True) -> int:
    return _ret(load().rra_finalize(), "rra_finalize", check)


def rra_allreduce(bufs, outs, count=None, dtype=None, op=RRA_SUM, algo=RRA_ALGO_AUTO, stream=None,
                  check=True, nranks=None) -> int:
    count, dtype = _resolve(bufs, count, dtype)
    n = len(bufs) if nranks is None else nranks
    st = load().rra_allreduce(_ptr_array(bufs), _ptr_array(outs), n, count, dtype, op, algo,
                              _stream(stream, bufs[0] if bufs else None))
    return _ret(st, "rra_allreduce", check)


def rra_allreduce_two_shot_static(bufs, outs, count=None, dtype=None, op=RRA_SUM, stream=None,
                                  check=True, nranks=None) -> int:
    """Two-shot all-reduce whose scratch is a static device array inside the
    library: no rra_init and no device allocation, for callers that may not
    allocate.  Calls that overlap on the GPU share that array and race."""
    count, dtype = _resolve(bufs, count, dtype)
    n = len(bufs) if nranks is None else nranks
    st = load().rra_allreduce_two_shot_static(_ptr_array(bufs), _ptr_array(outs), n, count, dtype, op,
                                              _stream(stream, bufs[0] if bufs else None))
    return _ret(st, "rra_allreduce_two_shot_static", check)


def rra_reduce_scatter(bufs, outs, recvcount=None, dtype=None, op=RRA_SUM, algo=RRA_ALGO_AUTO,
                       stream=None, check=True, nranks=None) -> int:
    if recvcount is None and outs and not isinstance(outs[0], int):
        recvcount = int(outs[0].numel())
    recvcount, dtype = _resolve(bufs, recvcount, dtype)
    n = len(bufs) if nranks is None else nranks
    st = load().rra_reduce_scatter(_ptr_array(bufs), _ptr_array(outs), n, recvcount, dtype, op, algo,
                                   _stream(stream, bufs[0] if bufs else None))
    return _ret(st, "rra_reduce_scatter", check)


def rra_all_gather(bufs, outs, sendcount=None, dtype=None, algo=RRA_ALGO_AUTO, stream=None,
                   check=True, nranks=None) -> int:
    sendcount, dtype = _resolve(bufs, sendcount, dtype)
    n = len(bufs) if nranks is None else nranks
    st = load().rra_all_gather(_ptr_array(bufs), _ptr_array(outs), n, sendcount, dtype, algo,
                               _stream(stream, bufs[0] if bufs else None))
    return _ret(st, "rra_all_gather", check)


def rra_allreduce_rmsnorm(bufs, outs, gamma, hidden, eps=1e-6, rows=None, dtype=None, stream=None,
                          check=True, nranks=None) -> int:
    count, dtype = _resolve(bufs, None if rows is None else rows * hidden, dtype)
    rows = count // hidden if rows is None else rows
    n = len(bufs) if nranks is None else nranks
    st = load().rra_allreduce_rmsnorm(_ptr_array(bufs), _ptr_array(outs), n, rows, hidden, _ptr(gamma),
                                      eps, dtype, _stream(stream, bufs[0] if bufs else None))
    return _ret(st, "rra_allreduce_rmsnorm", check)


def rra_ll_wire_bytes(payload_bytes: int) -> int:
    return int(load().rra_ll_wire_bytes(payload_bytes))


def rra_ll128_wire_bytes(payload_bytes: int) -> int:
    return int(load().rra_ll128_wire_bytes(payload_bytes))


def _nbytes(t):
    return int(t.numel() * t.element_size())


def rra_ll_pack(payload, wire, flag: int, payload_bytes=None, stream=None, check=True) -> int:
    B = _nbytes(payload) if payload_bytes is None else payload_bytes
    st = load().rra_ll_pack(_ptr(payload), B, _ptr(wire), flag, _stream(stream, payload))
    return _ret(st, "rra_ll_pack", check)


def rra_ll128_pack(payload, wire, flag: int, payload_bytes=None, stream=None, check=True) -> int:
    B = _nbytes(payload) if payload_bytes is None else payload_bytes
    st = load().rra_ll128_pack(_ptr(payload), B, _ptr(wire), flag, _stream(stream, payload))
    return _ret(st, "rra_ll128_pack", check)


def rra_ll_unpack(wires, out, expected_flag: int, dtype=None, payload_bytes=None, op=RRA_SUM,
                  stream=None, check=True, nsrc=None) -> int:
    dtype = _dtype_of(out) if dtype is None else dtype
    B = _nbytes(out) if payload_bytes is None else payload_bytes
    n = len(wires) if nsrc is None else nsrc
    st = load().rra_ll_unpack(_ptr_array(wires), n, _ptr(out), B, dtype, op, expected_flag,
                              _stream(stream, out))
    return _ret(st, "rra_ll_unpack", check)


def rra_ll128_unpack(wires, out, expected_flag: int, dtype=None, payload_bytes=None, op=RRA_SUM,
                     stream=None, check=True, nsrc=None) -> int:
    dtype = _dtype_of(out) if dtype is None else dtype
    B = _nbytes(out) if payload_bytes is None else payload_bytes
    n = len(wires) if nsrc is None else nsrc
    st = load().rra_ll128_unpack(_ptr_array(wires), n, _ptr(out), B, dtype, op, expected_flag,
                                 _stream(stream, out))
    return _ret(st, "rra_ll128_unpack", check)


def rra_query_status(stream=None):
    """Synchronize the stream and read/clear the device status.
    Returns (status, [code, rank, peer, index])."""
    info = (ctypes.c_int32 * 4)()
    st = load().rra_query_status(_stream(stream), info)
    return st, list(info)


def rra_query_status_static(stream=None):
    """Synchronize the stream and read/clear the status of
    rra_allreduce_two_shot_static (allocates nothing).
    Returns (status, [code, rank, peer, index])."""
    info = (ctypes.c_int32 * 4)()
    st = load().rra_query_status_static(_stream(stream), info)
    return st, list(info)


def rra_select_algo(nranks: int, bytes_per_rank: int, dtype: int) -> int:
    return int(load().rra_select_algo(nranks, bytes_per_rank, dtype))


def rra_load_tuning(path, check=True) -> int:
    p = None if path is None else os.fsencode(path)
    return _ret(load().rra_load_tuning(p), "rra_load_tuning", check)


def rra_set_timeout_ns(ns: int) -> None:
    load().rra_set_timeout_ns(ns)


def rra_debug_skip_rank(rank: int) -> None:
    load().rra_debug_skip_rank(rank)


def rra_set_max_ctas(max_ctas: int) -> None:
    load().rra_set_max_ctas(max_ctas)


def rra_dump_recent() -> str:
    buf = ctypes.create_string_buffer(64 * 256)
    load().rra_dump_recent(buf, len(buf))
    return buf.value.decode()
