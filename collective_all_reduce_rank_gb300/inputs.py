"""Seeded synthetic inputs for the virtual-rank collectives.

This module holds no arithmetic of the collectives: it only draws numbers.
Both the CPU oracle's tests and the CUDA path's tests and benchmark take
their inputs from here, so the two sides see identical data.

Recipe: numpy ``default_rng(seed)`` (PCG64), seed 0 unless stated; rank
buffers are drawn one after another from one generator, rank 0 first.
bfloat16 values are float32 draws rounded to nearest-even by torch's CPU
conversion and returned as their raw uint16 bits.

Workloads (message sizes are per rank):

* ``int8range`` -- integers uniform in [-8, 8] stored as float32 (exact in
  float32, so every summation order gives the same bits);
* ``ones``      -- all ones (the all-reduce sanity check: the sum is n);
* ``normal``    -- normal(0, sigma) (sigma = 1 for tensor-parallel
  activations, 1e-2 for gradient buckets);
* ``int20``     -- int32 uniform in [-2^20, 2^20].
"""
from __future__ import annotations

import numpy as np

NP_DTYPES = {"int32": np.int32, "float32": np.float32, "bfloat16": np.uint16}
ELEM_SIZE = {"int32": 4, "float32": 4, "bfloat16": 2}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits (round to nearest even) via torch's CPU cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def draw(rng: np.random.Generator, count: int, dtype: str, dist: str, sigma: float = 1.0):
    """One rank's buffer of ``count`` elements."""
    if dist == "ones":
        v = np.ones(count, dtype=np.float32)
    elif dist == "int8range":
        v = rng.integers(-8, 8, size=count, endpoint=True).astype(np.float32)
    elif dist == "normal":
        v = rng.normal(0.0, sigma, size=count).astype(np.float32)
    elif dist == "int20":
        v = rng.integers(-(1 << 20), 1 << 20, size=count, endpoint=True, dtype=np.int64)
        if dtype == "int32":
            return v.astype(np.int32)
        v = v.astype(np.float32)
    elif dist == "bits":
        # arbitrary bit patterns (int32 only): exercises wrap-around
        return rng.integers(-(1 << 31), (1 << 31) - 1, size=count, endpoint=True,
                            dtype=np.int64).astype(np.int32)
    else:
        raise ValueError(dist)
    if dtype == "int32":
        return v.astype(np.int32)
    if dtype == "float32":
        return v.astype(np.float32)
    if dtype == "bfloat16":
        return to_bf16_bits(v)
    raise ValueError(dtype)


def make_ranks(n: int, count: int, dtype: str, dist: str, seed: int = 0, sigma: float = 1.0):
    """n rank buffers of ``count`` elements each, drawn rank 0 first."""
    rng = np.random.default_rng(seed)
    return [draw(rng, count, dtype, dist, sigma) for _ in range(n)]


# --- the named workloads ---------------------------------------------------

def cfg_small_exact(seed: int = 0):
    """n=2 ranks, float32 SUM of 4096 integers in [-8, 8] per rank."""
    return make_ranks(2, 4096, "float32", "int8range", seed)


def cfg_sanity(n: int = 2):
    """ones(128) on every rank: the all-reduce must give n everywhere."""
    return make_ranks(n, 128, "float32", "ones")


TP_TOKENS = (1, 8, 32, 512)
TP_HIDDEN = 5120


def cfg_tp_activations(tokens: int, seed: int = 0):
    """n=8 ranks, bfloat16 activations [tokens, 5120], normal(0, 1)."""
    return make_ranks(8, tokens * TP_HIDDEN, "bfloat16", "normal", seed, 1.0)


BUCKET_COUNT = 25_000_000


def cfg_gradient_bucket(count: int = BUCKET_COUNT, seed: int = 0):
    """n=8 ranks, float32 gradient bucket of 25M elements, normal(0, 1e-2)."""
    return make_ranks(8, count, "float32", "normal", seed, 1e-2)


LL_SIZES = tuple(1 << k for k in range(10, 29))  # 1 KiB .. 256 MiB


def cfg_ll_payloads(payload_bytes: int, n: int = 4, seed: int = 0):
    """n=4 int32 payloads of payload_bytes bytes each, uniform in [-2^20, 2^20]."""
    return make_ranks(n, payload_bytes // 4, "int32", "int20", seed)


SWEEP_SIZES = tuple(1 << k for k in range(10, 31))  # 1 KiB .. 1 GiB per rank
SWEEP_RANKS = (2, 4, 8)


def cfg_sweep(n: int, bytes_per_rank: int, dtype: str, seed: int = 0):
    """Message-size sweep point: int32 in [-2^20, 2^20] or bfloat16 normal(0,1)."""
    count = bytes_per_rank // ELEM_SIZE[dtype]
    dist = "int20" if dtype == "int32" else "normal"
    return make_ranks(n, count, dtype, dist, seed, 1.0)


def counter_ints(rank: int, idx):
    """Counter-based integers in [-128, 128) for the element indices ``idx``
    (an int64 numpy array or torch tensor) of rank ``rank``: a buffer too
    large to draw and copy from the host is filled on the device with the
    same values the host computes for a sample of its indices.

    v = ((lo * 0x9E3779B1 + hi * 0x85EBCA77 + (rank + 1) * 0xC2B2AE3D) >> 15)
        mod 256 - 128, with lo = idx mod 2^20 and hi = idx >> 20: every term
    stays below 2^53 for idx < 2^34, so int64 arithmetic is exact on both
    sides, and indices 2^k apart (k >= 20) get unrelated values.  The values
    are exact in int32, float32 and bfloat16, and so is a sum of up to eight
    of them in int32 and float32."""
    lo = idx & 0xFFFFF
    hi = idx >> 20
    h = lo * 0x9E3779B1 + hi * 0x85EBCA77 + (rank + 1) * 0xC2B2AE3D
    return ((h >> 15) & 0xFF) - 128
