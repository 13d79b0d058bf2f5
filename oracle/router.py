"""Top-k softmax router (oracle).

FreeToken write-up, "decode co-design" section and Fig. 2 caption: per MoE
layer the GPU router picks the top-k of E routed experts for each token; the
layer output is the routing-weighted sum of the selected experts.

Readings where the pages are silent:
* selection is by logit, descending, ties going to the lower expert index;
* the weights are a softmax over the k selected logits (equivalently the
  full softmax renormalised over the selected experts), so each token's
  weights sum to 1;
* a NaN logit is treated as -inf (it is never preferred to a real logit);
* the weights use exp(l_j - l_max) with exp taken as 1 for every selected
  logit equal to the largest one, i.e. the limit of the softmax over equal
  logits: a token whose selected logits are all -inf (or NaN) gets equal
  weights 1/k, and the +inf entries of a token share its weight equally.
"""
from __future__ import annotations

import math

import numpy as np


def logits_from_router(x: np.ndarray, w_r: np.ndarray) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * W_r[e, h], in float64."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w_r, dtype=np.float64).T


def topk_ids(logits_row: np.ndarray, k: int) -> list[int]:
    """The k experts of one token in selection order."""
    vals = [(-np.inf if np.isnan(v) else float(v)) for v in logits_row]
    order = sorted(range(len(vals)), key=lambda e: (-vals[e], e))
    return order[:k]


def topk_softmax(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """ids int32 [B, k] and weights float64 [B, k] for logits [B, E]."""
    logits = np.asarray(logits, dtype=np.float64)
    B, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = np.zeros((B, k), dtype=np.int32)
    w = np.zeros((B, k), dtype=np.float64)
    for t in range(B):
        sel = topk_ids(logits[t], k)
        ids[t] = sel
        z = np.array([logits[t, e] for e in sel], dtype=np.float64)
        z = np.where(np.isnan(z), -np.inf, z)
        # z[0] is the largest selected logit; equal logits (also -inf == -inf
        # and +inf == +inf) contribute exp(0) = 1
        z = np.array([1.0 if zj == z[0] else math.exp(zj - z[0]) for zj in z])
        w[t] = z / z.sum()
    return ids, w


def topk_margin(logits: np.ndarray, k: int) -> float:
    """Smallest gap between the k-th and (k+1)-th largest logit over all tokens (inf if k == E)."""
    logits = np.asarray(logits, dtype=np.float64)
    if k >= logits.shape[1]:
        return float("inf")
    s = -np.sort(-logits, axis=1)
    return float(np.min(s[:, k - 1] - s[:, k]))
