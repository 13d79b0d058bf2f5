"""Pins for the oracle's cache simulator (oracle.lru).

The simulator picks victims for a whole call in one pass over stamps.  It is
checked against an independently written ordered-list LRU that processes the
call's distinct experts one by one (the classic move-to-front formulation of
"evict the expert not requested for the longest time"), exhaustively on tiny
traces and on random ones, plus the invariants the pages fix: a hit never
misses while resident, a cache that holds every (layer, expert) pair never
evicts, and GPU memory changes performance only.
"""
import itertools
import random

import numpy as np
import pytest

from oracle import lru


class ListLRU:
    """Brute-force LRU: an ordered list of keys, least recent first."""

    def __init__(self, L, E, C):
        self.L, self.E, self.C = L, E, C
        self.order = []
        self.slot = {}
        self.calls = 0

    def access(self, layer, ids):
        U = sorted(set(int(e) for e in np.asarray(ids).reshape(-1)))
        if len(U) > self.C:
            raise lru.CapacityError()
        keys = [layer * self.E + e for e in U]
        call_keys = set(keys)
        out = []
        for e, key in zip(U, keys):
            if key in self.slot:
                self.order.remove(key)
                self.order.append(key)
                out.append((self.calls, layer, e, lru.HIT, self.slot[key], -1))
                continue
            used = set(self.slot.values())
            free = [s for s in range(self.C) if s not in used]
            if free:
                s, ev = free[0], -1
            else:
                ev = next(k for k in self.order if k not in call_keys)
                self.order.remove(ev)
                s = self.slot.pop(ev)
            self.slot[key] = s
            self.order.append(key)
            out.append((self.calls, layer, e, lru.MISS, s, ev))
        self.calls += 1
        return out

    def resize(self, C_new):
        if C_new >= self.C:
            self.C = C_new
            return []
        keep = set(self.order[-C_new:]) if C_new > 0 else set()
        out = []
        for key, s in sorted(self.slot.items(), key=lambda kv: kv[1]):
            if key not in keep:
                out.append((self.calls, key // self.E, key % self.E, lru.RESIZE_EVICT, s, key))
        for _, _, _, _, s, key in out:
            del self.slot[key]
            self.order.remove(key)
        used = set(self.slot.values())
        vacant = [s for s in range(C_new) if s not in used]
        movers = sorted((s, k) for k, s in self.slot.items() if s >= C_new)
        for (s, k), d in zip(movers, vacant):
            self.slot[k] = d
        self.C = C_new
        return out


    def prefill(self, l0, l1, chunks=1):
        """Physical model: the buffers are the last 2E slots; each layer's
        experts are requested in ascending order, each either read where it
        is resident or copied into its buffer slot, replacing that slot's
        content; a requested expert becomes the most recent."""
        E, C = self.E, self.C
        buf0 = C - 2 * E
        out = []
        for key, s in sorted(self.slot.items(), key=lambda kv: kv[1]):
            if s >= buf0:
                out.append((self.calls, key // E, key % E, lru.PREFILL_EVICT, s, key))
        for _, _, _, _, s, key in out:
            del self.slot[key]
            self.order.remove(key)
        table = []
        for i in range(chunks * (l1 - l0)):
            layer = l0 + i % (l1 - l0)
            row = []
            for e in range(E):
                key = layer * E + e
                if key not in self.slot:
                    s = buf0 + (i % 2) * E + e
                    for k in [k for k, v in self.slot.items() if v == s]:
                        del self.slot[k]
                        self.order.remove(k)
                    self.slot[key] = s
                else:
                    self.order.remove(key)
                self.order.append(key)
                row.append(self.slot[key])
            table.append(row)
        return out, table


def run_both(L, E, C, trace):
    a, b = lru.CacheSim(L, E, C), ListLRU(L, E, C)
    ea, eb = [], []
    for layer, ids in trace:
        if layer == "prefill":
            ev, ta = a.prefill(*ids)
            evb, tb = b.prefill(*ids)
            ea += [e.as_tuple() for e in ev]
            eb += evb
            assert ta.tolist() == tb
            continue
        try:
            ev, _ = a.access(layer, ids)
            ea += [e.as_tuple() for e in ev]
        except lru.CapacityError:
            ea.append("cap")
        try:
            eb += b.access(layer, ids)
        except lru.CapacityError:
            eb.append("cap")
    return ea, eb


def test_exhaustive_single_layer_k1():
    # every trace of length 6 over 3 experts, one expert per call, C = 1..3
    for C in (1, 2, 3):
        for seq in itertools.product(range(3), repeat=6):
            trace = [(0, np.array([[e]])) for e in seq]
            ea, eb = run_both(1, 3, C, trace)
            assert ea == eb, (C, seq)


def test_exhaustive_two_layers_k2():
    # two layers alternating, two experts routed per call out of 3, C = 2..4
    pairs = [(0, 1), (0, 2), (1, 2), (1, 1), (2, 0)]
    for C in (2, 3, 4):
        for seq in itertools.product(range(len(pairs)), repeat=4):
            trace = [(i % 2, np.array([pairs[p]])) for i, p in enumerate(seq)]
            ea, eb = run_both(2, 3, C, trace)
            assert ea == eb, (C, seq)


@pytest.mark.parametrize("seed", range(6))
def test_random_traces(seed):
    rng = random.Random(seed)
    L, E = 3, 10
    C = rng.choice([4, 7, 12, 30])
    trace = []
    for _ in range(300):
        B, k = rng.choice([(1, 2), (2, 2), (3, 1), (2, 3)])
        trace.append((rng.randrange(L), np.array([[rng.randrange(E) for _ in range(k)] for _ in range(B)])))
    ea, eb = run_both(L, E, C, trace)
    assert ea == eb


def test_resize_matches_list_truncation():
    rng = random.Random(3)
    L, E, C = 2, 12, 10
    a, b = lru.CacheSim(L, E, C), ListLRU(L, E, C)
    for phase, C_new in enumerate([10, 4, 9, 3, 3, 11]):
        if phase:
            ra = [e.as_tuple() for e in a.resize(C_new)]
            rb = b.resize(C_new)
            assert ra == rb
            assert {k: s for s, k in enumerate(a.owner) if k >= 0} == b.slot
        for _ in range(60):
            layer = rng.randrange(L)
            ids = np.array([[rng.randrange(E), rng.randrange(E)]])
            ev, _ = a.access(layer, ids)
            assert [e.as_tuple() for e in ev] == b.access(layer, ids)


def test_resize_keeps_most_recent_and_preserves_stamps():
    sim = lru.CacheSim(1, 8, 6)
    for e in [0, 1, 2, 3, 4, 5, 1, 3]:
        sim.access(0, np.array([[e]]))
    stamps = {int(k): int(sim.stamp[s]) for s, k in enumerate(sim.owner) if k >= 0}
    g = sim.g
    ev = sim.resize(3)
    assert sim.resident_keys() == {3, 1, 5}
    assert [e.expert for e in ev] == [0, 2, 4]  # ascending slot order: slots 0, 2, 4
    assert sim.g == g
    for s, k in enumerate(sim.owner):
        if k >= 0:
            assert int(sim.stamp[s]) == stamps[int(k)]
            assert sim.map[k] == s


def test_all_resident_means_no_miss():
    rng = np.random.default_rng(0)
    sim = lru.CacheSim(2, 16, 10)
    for _ in range(200):
        layer = int(rng.integers(2))
        ids = rng.integers(0, 16, size=(2, 2))
        resident = set(int(k) for k in sim.owner if k >= 0)
        keys = {layer * 16 + int(e) for e in ids.reshape(-1)}
        ev, _ = sim.access(layer, ids)
        if keys <= resident:
            assert all(e.kind == lru.HIT for e in ev)


def test_full_capacity_never_evicts():
    rng = np.random.default_rng(1)
    L, E = 3, 8
    sim = lru.CacheSim(L, E, L * E)
    for _ in range(400):
        ev, _ = sim.access(int(rng.integers(L)), rng.integers(0, E, size=(3, 2)))
        assert all(e.evicted_key == -1 for e in ev)


def test_capacity_error_leaves_state_unchanged():
    sim = lru.CacheSim(1, 8, 2)
    sim.access(0, np.array([[1, 2]]))
    snap = (sim.map.copy(), sim.owner.copy(), sim.stamp.copy(), sim.g, sim.calls)
    with pytest.raises(lru.CapacityError):
        sim.access(0, np.array([[3, 4], [5, 3]]))
    assert (sim.map == snap[0]).all() and (sim.owner == snap[1]).all() and (sim.stamp == snap[2]).all()
    assert (sim.g, sim.calls) == snap[3:]


def test_hand_worked_trace():
    # C = 2, one layer, experts: 0, 1, 0, 2, 1.
    # call0: 0 miss -> slot 0; call1: 1 miss -> slot 1; call2: 0 hit;
    # call3: 2 miss, LRU is 1 (slot 1); call4: 1 miss, LRU is 0 (slot 0).
    sim = lru.CacheSim(1, 4, 2)
    got = []
    for e in [0, 1, 0, 2, 1]:
        ev, slots = sim.access(0, np.array([[e]]))
        got += [(x.kind, x.slot, x.evicted_key) for x in ev]
    assert got == [(1, 0, -1), (1, 1, -1), (0, 0, -1), (1, 1, 1), (1, 0, 0)]
    assert lru.hit_rate([lru.Event(0, 0, 0, k, 0, -1) for k in (0, 0, 1, 0)]) == 0.75


def test_slot_ids_rewrite():
    sim = lru.CacheSim(1, 8, 4)
    ids = np.array([[5, 2], [2, 7]])
    ev, slots = sim.access(0, ids)
    slot_of = {e.expert: e.slot for e in ev}
    assert (slots == np.vectorize(slot_of.get)(ids)).all()


# ------------------------------------------------------------------ prefill --

def recency_order(sim):
    occ = [s for s in range(sim.C) if sim.owner[s] >= 0]
    return [int(sim.owner[s]) for s in sorted(occ, key=lambda s: int(sim.stamp[s]))]


@pytest.mark.parametrize("seed", range(40))
def test_prefill_matches_physical_model_inside_random_traces(seed):
    rng = random.Random(seed)
    L, E = 4, 3
    C = rng.randint(2 * E, L * E)
    trace = []
    for _ in range(rng.randint(3, 9)):
        if rng.random() < 0.3:
            l0 = rng.randint(0, L - 1)
            trace.append(("prefill", (l0, rng.randint(l0 + 1, L), rng.choice([1, 1, 2, 3]))))
        else:
            trace.append((rng.randint(0, L - 1), [[rng.randint(0, E - 1) for _ in range(2)]]))
    a, b = lru.CacheSim(L, E, C), ListLRU(L, E, C)
    ea, eb = [], []
    for layer, ids in trace:
        if layer == "prefill":
            ev, ta = a.prefill(*ids)
            evb, tb = b.prefill(*ids)
            assert ta.tolist() == tb
            ea += [e.as_tuple() for e in ev]
            eb += evb
        else:
            ev, _ = a.access(layer, ids)
            ea += [e.as_tuple() for e in ev]
            eb += b.access(layer, ids)
        # same residency, same slots, same recency order after every operation
        assert {int(a.owner[s]): s for s in range(C) if a.owner[s] >= 0} == b.slot
        assert recency_order(a) == b.order
        for key in range(L * E):
            assert (a.map[key] >= 0) == (key in b.slot)
    assert ea == eb


def test_prefill_survivors_seed_decode():
    # a full-model prefill on an empty cache leaves the last two layers' whole
    # expert sets resident in the buffers, so decode on those layers never misses
    L, E, k = 5, 8, 3
    sim = lru.CacheSim(L, E, 2 * E + 4)
    ev, table = sim.prefill(0, L)
    assert ev == []
    buf0 = sim.C - 2 * E
    assert table[L - 1].tolist() == [buf0 + ((L - 1) % 2) * E + e for e in range(E)]
    assert sim.resident_keys() == {l * E + e for l in (L - 2, L - 1) for e in range(E)}
    rng = np.random.default_rng(0)
    for layer in (L - 2, L - 1):
        ids = rng.choice(E, size=(2, k), replace=True)
        evs, _ = sim.access(layer, ids)
        assert all(e.kind == lru.HIT for e in evs)


def test_prefill_reads_resident_experts_in_place_and_keeps_one_copy():
    L, E = 3, 4
    sim = lru.CacheSim(L, E, 2 * E + 2)
    sim.access(1, np.array([[2, 3]]))  # layer 1's experts 2 and 3 land in slots 0 and 1
    assert sim.map[1 * E + 2] == 0 and sim.map[1 * E + 3] == 1
    ev, table = sim.prefill(0, L)
    assert table[1].tolist()[2:] == [0, 1]  # read where they are, not streamed
    keys = [int(k) for k in sim.owner if k >= 0]
    assert len(keys) == len(set(keys))
    assert sim.g == 2 + L * E


def test_prefill_carves_buffers_and_logs_evictions():
    L, E = 2, 2
    sim = lru.CacheSim(L, E, 5)
    sim.access(0, np.array([[0, 1]]))
    sim.access(1, np.array([[0, 1]]))
    sim.access(0, np.array([[0]]))  # hit; slots: 0->key0, 1->key1, 2->key2, 3->key3
    ev, _ = sim.prefill(1, 2)
    # buffers are slots 1..4: keys 1, 2, 3 evicted in slot order; key 0 stays
    assert [(e.slot, e.evicted_key, e.kind) for e in ev] == [(1, 1, lru.PREFILL_EVICT), (2, 2, lru.PREFILL_EVICT),
                                                             (3, 3, lru.PREFILL_EVICT)]
    assert sim.map[0] == 0
    with pytest.raises(lru.CapacityError):
        lru.CacheSim(L, E, 3).prefill(0, 1)


@pytest.mark.parametrize("seed", range(20))
def test_on_demand_prefill_matches_list_lru_in_chunks(seed):
    rng = random.Random(seed)
    L, E = 3, 6
    C = rng.randint(1, 2 * E - 1)
    a, b = lru.CacheSim(L, E, C), ListLRU(L, E, C)
    for _ in range(6):
        layer = rng.randrange(L)
        if rng.random() < 0.5:  # a prefill layer: many tokens routed
            ids = np.array([[rng.randrange(E) for _ in range(2)] for _ in range(rng.randint(1, 8))])
            ev, slot_of = a.prefill_on_demand(layer, ids)
            U = sorted(set(ids.reshape(-1).tolist()))
            evb = []
            for c0 in range(0, len(U), C):  # the list LRU, chunk by chunk
                evb += b.access(layer, np.array([U[c0:c0 + C]]))
            assert [e.as_tuple() for e in ev] == evb
            assert set(slot_of) == set(U)
        else:
            ids = np.array([[rng.randrange(E)]])
            assert [e.as_tuple() for e in a.access(layer, ids)[0]] == b.access(layer, ids)


def test_on_demand_prefill_is_one_call_when_the_layer_fits():
    sim, ref = lru.CacheSim(2, 8, 10), lru.CacheSim(2, 8, 10)
    ids = np.array([[3, 1], [1, 7], [5, 3]])
    ev, slot_of = sim.prefill_on_demand(1, ids)
    ev2, _ = ref.access(1, ids)
    assert [e.as_tuple() for e in ev] == [e.as_tuple() for e in ev2] and sim.calls == 1
    assert sorted(slot_of) == [1, 3, 5, 7]
