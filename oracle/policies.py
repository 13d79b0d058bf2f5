"""Expert placement policies replayed on one routing trace (CPU analysis).

TEST AND ANALYSIS INFRASTRUCTURE ONLY, like the rest of this package: plain
Python simulators that count decode-time expert misses; nothing on the GPU
path calls them.

FreeToken write-up, experimental results, expert-locality paragraph (the
Fig. 4b replay): the same routing traces are replayed at equal cache capacity
under FreeToken's global LRU over all layers, KTransformers' placement
refreshed from prefill routing, and llama.cpp's routing-agnostic static
split; the "Luce Spark" post adds calibrated pinning of the most used
(layer, expert) pairs plus a bounded ring of spare slots managed LRU.

Readings (the pages name the policies and describe their behaviour, not
their code; each is the plainest deterministic version of that description):
* A trace is a prompt of T_p tokens followed by T_d decode tokens of the
  same routing process.  Only decode accesses are counted; the prompt is
  what each policy may learn from.
* Accesses: per decode step and layer, the distinct experts routed by the
  step's tokens (the per-layer dedup of the cache control step), in
  ascending expert order.  Miss rate = misses / accesses.
* global_lru: the shared all-layer cache of capacity C with the victim rule
  of lru.CacheSim (empty slots first, then least recently stamped, never an
  expert of the same call), fed the prompt's accesses step by step first.
* prefill_placement: after the prompt, the C (layer, expert) pairs routed to
  most often during the prompt are resident (ties to the lower key); decode
  never changes the placement and a miss is not cached.
* static_split: whole layers resident regardless of routing, the last
  floor(C / E) layers (llama.cpp keeps the chosen layers' expert weights on
  the CPU), plus the lowest C mod E experts of the layer before them.
* pinned_ring: the C - R pairs routed to most often during the prompt are
  pinned; the remaining R = max(1, ceil(C / 8)) slots form a ring that
  caches cold experts under the same LRU rule (a call whose cold experts
  outnumber the ring admits the first R of them in ascending order).
"""
from __future__ import annotations

import math
from collections import OrderedDict

import numpy as np

from . import router


def step_accesses(ids_step: np.ndarray) -> list[int]:
    """Distinct experts of one (step, layer) call, ascending."""
    return sorted(set(int(e) for e in np.asarray(ids_step).reshape(-1)))


class LruCount:
    """Global LRU with the simulator's victim rule, counting misses only.

    An OrderedDict keeps keys least recent first; a call's distinct experts are
    stamped in ascending order (hits and misses alike), and a miss takes a free
    slot while any is left, else the least recent key not used by this call.
    """

    def __init__(self, C: int):
        self.C = C
        self.order: OrderedDict[int, None] = OrderedDict()

    def call(self, keys: list[int]) -> int:
        if len(keys) > self.C:
            raise ValueError("a call routes more distinct experts than there are slots")
        ks = set(keys)
        misses = 0
        for key in keys:
            if key in self.order:
                self.order.move_to_end(key)
                continue
            misses += 1
            if len(self.order) >= self.C:
                victim = next(k for k in self.order if k not in ks)
                del self.order[victim]
            self.order[key] = None
        return misses


def routed_ids(logits: np.ndarray, k: int) -> np.ndarray:
    """ids int [T, L, B, k] for logits [T, L, B, E]."""
    T, L, B, E = logits.shape
    out = np.zeros((T, L, B, k), dtype=np.int64)
    for t in range(T):
        for l in range(L):
            out[t, l], _ = router.topk_softmax(logits[t, l].astype(np.float64), k)
    return out


def prompt_counts(ids: np.ndarray, E: int) -> np.ndarray:
    """Routed (token, rank) pairs per key l*E + e over a prompt ids [T, L, B, k]."""
    T, L, B, k = ids.shape
    cnt = np.zeros(L * E, dtype=np.int64)
    for l in range(L):
        np.add.at(cnt, l * E + ids[:, l].reshape(-1), 1)
    return cnt


def most_used(cnt: np.ndarray, n: int) -> set[int]:
    """The n keys with the largest counts, ties to the lower key."""
    order = sorted(range(len(cnt)), key=lambda key: (-int(cnt[key]), key))
    return set(order[:max(0, n)])


def replay(ids: np.ndarray, T_p: int, E: int, C: int, policy: str) -> tuple[int, int]:
    """(misses, accesses) over the decode steps T_p .. T-1 of ids [T, L, B, k]."""
    T, L, B, k = ids.shape
    misses = accesses = 0
    if policy == "global_lru":
        cache = LruCount(C)
        for t in range(T):
            for l in range(L):
                keys = [l * E + e for e in step_accesses(ids[t, l])]
                m = cache.call(keys)
                if t >= T_p:
                    misses += m
                    accesses += len(keys)
        return misses, accesses
    if policy == "prefill_placement":
        resident = most_used(prompt_counts(ids[:T_p], E), C)
        ring = None
    elif policy == "static_split":
        full = min(L, C // E)
        resident = {l * E + e for l in range(L - full, L) for e in range(E)}
        if full < L:
            resident |= {(L - full - 1) * E + e for e in range(C - full * E)}
        ring = None
    elif policy == "pinned_ring":
        R = max(1, math.ceil(C / 8))
        resident = most_used(prompt_counts(ids[:T_p], E), C - R)
        ring = LruCount(R)
    else:
        raise ValueError(policy)
    for t in range(T_p, T):
        for l in range(L):
            keys = [l * E + e for e in step_accesses(ids[t, l])]
            accesses += len(keys)
            cold = [key for key in keys if key not in resident]
            if ring is None:
                misses += len(cold)
            else:
                admit = cold[:ring.C]
                misses += ring.call(admit) + (len(cold) - len(admit))
    return misses, accesses


POLICIES = ("global_lru", "prefill_placement", "static_split", "pinned_ring")
