"""Grouping of (token, rank) pairs by expert (oracle).

The layer evaluates the selected experts as one grouped FFN over the set
G = H ∪ F (FreeToken write-up, "measured bandwidths decide the split" section:
"grouped evaluation of G"); the tokens routed to each expert are gathered
together first.  Reading: the pairs are ordered by a *stable* sort of the flat
routed ids, so pairs of one expert keep ascending flat index t*k + j.
"""
from __future__ import annotations

import numpy as np


def permutation(ids: np.ndarray, E: int) -> tuple[np.ndarray, np.ndarray]:
    """perm int32 [B*k] (flat pair indices grouped by expert) and offsets int32 [E+1]."""
    flat = np.asarray(ids).reshape(-1)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return perm, offsets
