"""Cost model and bandwidth metrics as the pages state them (oracle side).

Test infrastructure only, like the rest of ``oracle/``.

* alpha-beta time of one all-reduce of S bytes per GPU over n GPUs, from
  "Collective communication: NCCL's algorithms and protocols, and custom
  all-reduce in inference frameworks", section "Algorithms: the ways to run
  one all-reduce" (the table of formulas for ring, tree, one-shot, two-shot
  and NVLS);
* the one-shot / two-shot crossover of the same page, "Exercises", 2;
* algbw = S / t and busbw = algbw x factor, with factor 2(n-1)/n for
  all-reduce, (n-1)/n for all-gather and reduce-scatter and 1 for broadcast,
  from the same page, section "Reading nccl-tests".
"""
from __future__ import annotations

import math

ALGOS = ("ring", "tree", "one-shot", "two-shot", "NVLS")


def ab_time(algo: str, n: int, S: float, alpha: float, beta: float) -> float:
    """Seconds for an all-reduce of S bytes per GPU under the alpha-beta model."""
    if algo == "ring":
        return 2 * (n - 1) * alpha + 2 * (n - 1) / n * S / beta
    if algo == "tree":
        return 2 * math.log2(n) * alpha + 2 * S / beta
    if algo == "one-shot":
        return 2 * alpha + (n - 1) * S / beta
    if algo == "two-shot":
        return 4 * alpha + 2 * (n - 1) / n * S / beta
    if algo == "NVLS":
        return 2 * alpha + S / beta
    raise ValueError(algo)


def oneshot_twoshot_crossover(n: int, alpha: float, beta: float) -> float | None:
    """Message size S* where one-shot and two-shot cost the same; None when
    the denominator vanishes (n = 2: one-shot is never worse)."""
    den = (n - 1) * (1 - 2 / n)
    if den == 0:
        return None
    return 2 * alpha * beta / den


def bus_factor(collective: str, n: int) -> float:
    if collective == "allreduce":
        return 2 * (n - 1) / n
    if collective in ("allgather", "reducescatter"):
        return (n - 1) / n
    if collective == "broadcast":
        return 1.0
    raise ValueError(collective)


def algbw(S: float, t: float) -> float:
    return S / t


def busbw(collective: str, n: int, S: float, t: float) -> float:
    return algbw(S, t) * bus_factor(collective, n)
