"""Bandwidth-adaptive fill count q* (oracle).

FreeToken write-up, "measured bandwidths decide the split" section: with m
distinct missed experts of S bytes, pinned-memory transfer bandwidth B_P and
host expert-processing bandwidth B_H, a saturated link leaves
B_R = max(B_H - B_P, 0) for CPU execution; T_fill(q) ~ qS/B_P and
T_cpu(m-q) ~ (m-q)S/(B_H - B_P); balancing the two gives q* ~ m * B_P / B_H.
In practice q* is rounded to an integer and at least one fill is kept so the
cache keeps warming.

Readings: rounding is to the nearest integer (halves away from zero), the
result is clamped to [1, m] when m >= 1, and q* = 0 when m = 0.
"""
from __future__ import annotations

import math


def qstar(m: int, b_p: float, b_h: float) -> int:
    if m <= 0:
        return 0
    if b_h <= b_p:  # no residual host bandwidth: pure on-demand fill
        return m
    q = math.floor(m * b_p / b_h + 0.5)
    return max(1, min(m, q))


def branch_times(m: int, q: int, S: float, b_p: float, b_h: float) -> tuple[float, float]:
    """(T_fill, T_cpu) for q fills and m - q CPU experts."""
    t_fill = q * S / b_p
    b_r = max(b_h - b_p, 0.0)
    if m - q <= 0:
        t_cpu = 0.0
    else:
        t_cpu = (m - q) * S / b_r if b_r > 0 else float("inf")
    return t_fill, t_cpu
