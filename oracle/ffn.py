"""SwiGLU expert FFN and the routed MoE layer output (oracle).

FreeToken write-up: each selected expert is evaluated on the tokens routed to
it; decode is memory-bound, reading each routed expert's weights once per
token ("decode: cache misses and the CPU bandwidth limit" section); the GPU
and CPU partial sums merge exactly, with no algorithmic approximation (Fig. 2
caption, "measured bandwidths decide the split" section), so caching changes
where weights are read, never the result.

Per expert: h = SiLU(x W_gate^T) * (x W_up^T); o = h W_down^T, with
SiLU(z) = z / (1 + exp(-z)).  Layer: y_t = sum_j w_tj * o_tj (+ the shared
expert's output with weight 1).  Readings: the shared expert is ungated; the
sum over j runs in rank order.  All arithmetic here is float64.
"""
from __future__ import annotations

import numpy as np


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def expert(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """SwiGLU expert on x [n, H] -> [n, H] (float64)."""
    x = np.asarray(x, dtype=np.float64)
    h = silu(x @ w_gate.T) * (x @ w_up.T)
    return h @ w_down.T


def moe_layer(x: np.ndarray, ids: np.ndarray, w: np.ndarray, get_expert, shared=None) -> np.ndarray:
    """y [B, H] = sum_j w[t, j] * expert_{ids[t, j]}(x_t) (+ shared(x_t)).

    get_expert(e) -> (W_gate, W_up, W_down) for routed expert e of this layer;
    shared is None or such a triple.
    """
    x = np.asarray(x, dtype=np.float64)
    B, H = x.shape
    y = np.zeros((B, H), dtype=np.float64)
    cache = {}
    for t in range(B):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = get_expert(e)
            y[t] += float(w[t, j]) * expert(x[t:t + 1], *cache[e])[0]
        if shared is not None:
            y[t] += expert(x[t:t + 1], *shared)[0]
    return y


def dense_layer(x: np.ndarray, gates: np.ndarray, get_expert, E: int, shared=None) -> np.ndarray:
    """All-experts-resident evaluation: y_t = sum_e gates[t, e] * expert_e(x_t) (+ shared)."""
    x = np.asarray(x, dtype=np.float64)
    y = np.zeros_like(x)
    for e in range(E):
        g = gates[:, e]
        if np.any(g != 0):
            y += g[:, None] * expert(x, *get_expert(e))
    if shared is not None:
        y += expert(x, *shared)
    return y
