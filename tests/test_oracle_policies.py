"""Pins for the placement-policy replay (oracle.policies): each policy on a
hand-worked trace, the fast miss-counting LRU against the cache simulator,
and closed forms (a routing-agnostic static split misses the non-resident
share of uniformly spread accesses; every policy stops missing once the
whole pool fits)."""
import random

import numpy as np
import pytest

from oracle import lru, policies


def hand_trace():
    # L = 2 layers, E = 3 experts, k = 1, B = 1; prompt = steps 0..1, decode = steps 2..5
    per_step = [(0, 1), (0, 2), (1, 1), (0, 2), (1, 1), (2, 2)]
    return np.array([[[[a]], [[b]]] for a, b in per_step], dtype=np.int64)  # [T, L, B, k]


@pytest.mark.parametrize("policy,misses", [("global_lru", 2), ("prefill_placement", 1), ("static_split", 3),
                                           ("pinned_ring", 2)])
def test_policies_on_a_hand_worked_trace(policy, misses):
    # worked by hand at C = 4 (keys l*3 + e; prompt counts: key 0 twice, keys 4 and 5 once):
    # LRU fills 0,4,5 in the prompt, takes the free slot for 1 and later evicts 0 for 2;
    # prefill placement keeps {0, 4, 5, 1} and misses only expert 2 of layer 0;
    # the static split keeps layer 1 and expert 0 of layer 0 and misses 1, 1, 2;
    # pinning keeps {0, 4, 5} and its one-slot ring misses 1 once, then 2
    assert policies.replay(hand_trace(), 2, 3, 4, policy) == (misses, 8)


@pytest.mark.parametrize("seed", range(30))
def test_lru_counter_matches_the_cache_simulator(seed):
    rng = random.Random(seed)
    L, E = 3, 5
    C = rng.randint(3, L * E)
    sim, fast = lru.CacheSim(L, E, C), policies.LruCount(C)
    for _ in range(40):
        layer = rng.randrange(L)
        ids = np.array([[rng.randrange(E) for _ in range(rng.randint(1, 3))]])
        keys = [layer * E + e for e in policies.step_accesses(ids)]
        ev, _ = sim.access(layer, ids)
        assert fast.call(keys) == sum(1 for e in ev if e.kind == lru.MISS)
        assert set(fast.order) == sim.resident_keys()


def test_static_split_misses_the_non_resident_share():
    rng = np.random.default_rng(0)
    T, L, E, k = 400, 8, 16, 1
    ids = rng.integers(0, E, size=(T, L, 1, k))
    for C in (16, 48, 100):
        m, a = policies.replay(ids, 0, E, C, "static_split")
        assert abs(m / a - (1 - C / (L * E))) < 0.03


@pytest.mark.parametrize("policy", policies.POLICIES)
def test_whole_pool_resident_never_misses_after_the_prompt(policy):
    rng = np.random.default_rng(1)
    T, L, E, k = 60, 3, 4, 2
    ids = rng.integers(0, E, size=(T, L, 1, k))
    ids[:4, :, 0, 0] = np.arange(E)[:, None]   # the prompt routes to every expert once
    m, a = policies.replay(ids, 4, E, L * E + (L * E + 7) // 8, policy)
    assert m == 0 and a > 0
