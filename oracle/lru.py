"""Shared all-layer LRU expert cache (oracle simulator).

FreeToken write-up, "router-following LRU cache" and "CUDA Graph-compatible LRU
cache" sections:
* one GPU expert cache shared by every MoE layer; a slot holds one
  (layer, expert) pair, addressed by the flat key ``l*E + e``;
* a hit refreshes the expert's recency, a fill admits the newly selected
  expert, an eviction removes the expert the model has not asked for for the
  longest time;
* per layer one pass deduplicates the routed experts, classifies them against
  the residency table, picks K victim slots at once (the miss path takes the
  first q <= K of them) and rewrites logical ids to slot ids.
"Elastic memory management" section: at a safe point the cache is rebuilt to
a new slot budget without touching the host pool.  "Full-layer double
buffering" section: prefill carves two full-layer buffers out of the same
slot pool, streams each layer's whole expert set into one of them while the
previous layer computes on the other, and whatever survives prefill seeds
the decode cache (there is no separate prefill cache and no hand-off step).

Readings where the pages are silent (each one is a plain deterministic choice):
* U = the sorted distinct experts routed by the B tokens of the call.  Every
  member of U is classified against the state *before* the call.
* Recency is a stamp from a global counter g: the member of U with rank r gets
  stamp g + r, hit or miss; then g += |U|.  Stamps are unique.
* Victims: among slots not holding a hit of this call, empty slots come first
  (lowest index first), then occupied slots by ascending stamp.  The i-th miss
  in ascending expert order takes the i-th victim.  A miss never evicts an
  expert routed in the same call.
* |U| > C is a capacity error and leaves the state unchanged.
* Resize to C' < C keeps the C' most recently used experts; the others are
  evicted in ascending slot order; survivors sitting in slots >= C' move, in
  ascending old-slot order, into the vacant slots < C' in ascending order.
  Growing appends empty slots.  Stamps, the map and g are preserved.
* Prefill over layers l0 .. l1-1 (needs C >= 2E): the buffers are the last
  2E slots; buffer b = slots C-2E+b*E .. C-2E+b*E+E-1, expert e of a layer
  in buffer b sits at slot C-2E+b*E+e.  First every entry in the buffers is
  evicted (PREFILL_EVICT events, ascending slot).  Then step i (layer
  l0 + i mod (l1-l0); a long prompt repeats the layers once per chunk) uses
  buffer i mod 2: every expert e of the layer, in ascending order, is either
  already resident in a slot outside the buffers (read in place, no copy) or
  streamed into its buffer slot (whatever that slot held is dropped); either
  way its stamp becomes g + e, then g += E.  The buffer slots keep what was
  last streamed into them: after prefill they are ordinary cache entries, so
  the last two layers' streamed experts seed decode.
* Prefill with C < 2E (the pages' on-demand fallback, no oversubscription):
  per layer, the distinct routed experts in ascending order are accessed in
  consecutive chunks of at most C, each chunk exactly like one decode call.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

HIT, MISS, RESIZE_EVICT, PREFILL_EVICT = 0, 1, 2, 3


class CapacityError(RuntimeError):
    pass


@dataclass(frozen=True)
class Event:
    call: int
    layer: int
    expert: int
    kind: int
    slot: int
    evicted_key: int  # -1 if none

    def as_tuple(self):
        return (self.call, self.layer, self.expert, self.kind, self.slot, self.evicted_key)


class CacheSim:
    """Stamp-based simulator of the shared expert cache's bookkeeping."""

    def __init__(self, L: int, E: int, C: int):
        if C < 0:
            raise ValueError("C >= 0")
        self.L, self.E, self.C = L, E, C
        self.map = np.full(L * E, -1, dtype=np.int64)
        self.owner = np.full(C, -1, dtype=np.int64)
        self.stamp = np.zeros(C, dtype=np.uint64)
        self.g = 0
        self.calls = 0

    # -- one layer call ------------------------------------------------------
    def access(self, layer: int, ids: np.ndarray) -> tuple[list[Event], np.ndarray]:
        """Process the routed ids [B, k] of one layer call.

        Returns the events (one per distinct expert, ascending expert order)
        and slot_ids [B, k] (the logical ids rewritten to slot ids).
        """
        E = self.E
        ids = np.asarray(ids)
        U = sorted(set(int(e) for e in ids.reshape(-1)))
        if len(U) > self.C:
            raise CapacityError(f"{len(U)} distinct experts > {self.C} slots")
        call = self.calls
        keys = [layer * E + e for e in U]
        hit_slot = {key: int(self.map[key]) for key in keys if self.map[key] >= 0}
        taken = set(hit_slot.values())
        misses = [key for key in keys if key not in hit_slot]
        victims = []
        if misses:
            # order the candidate slots by (0, slot) if empty else (1, stamp)
            slots = np.arange(self.C)
            cand = slots[~np.isin(slots, list(taken))]
            occupied = (self.owner[cand] >= 0).astype(np.int64)
            secondary = np.where(occupied == 1, self.stamp[cand].astype(np.int64), cand)
            order = np.lexsort((secondary, occupied))
            victims = [int(s) for s in cand[order][:len(misses)]]
        events, slot_of = [], {}
        mi = 0
        for r, (e, key) in enumerate(zip(U, keys)):
            if key in hit_slot:
                s = hit_slot[key]
                self.stamp[s] = np.uint64(self.g + r)
                events.append(Event(call, layer, e, HIT, s, -1))
            else:
                s = victims[mi]
                mi += 1
                ev = int(self.owner[s])
                if ev >= 0:
                    self.map[ev] = -1
                self.map[key] = s
                self.owner[s] = key
                self.stamp[s] = np.uint64(self.g + r)
                events.append(Event(call, layer, e, MISS, s, ev))
            slot_of[e] = s
        self.g += len(U)
        self.calls += 1
        slot_ids = np.vectorize(lambda e: slot_of[int(e)], otypes=[np.int64])(ids) if ids.size else ids
        return events, slot_ids

    # -- safe-point resize ---------------------------------------------------
    def resize(self, C_new: int) -> list[Event]:
        """Rebuild the cache with C_new slots; returns RESIZE_EVICT events (ascending slot)."""
        C = self.C
        events = []
        if C_new >= C:
            self.owner = np.concatenate([self.owner, np.full(C_new - C, -1, dtype=np.int64)])
            self.stamp = np.concatenate([self.stamp, np.zeros(C_new - C, dtype=np.uint64)])
            self.C = C_new
            return events
        occupied = [s for s in range(C) if self.owner[s] >= 0]
        by_recency = sorted(occupied, key=lambda s: -int(self.stamp[s]))
        keep = set(by_recency[:C_new])
        for s in sorted(occupied):
            if s not in keep:
                key = int(self.owner[s])
                events.append(Event(self.calls, key // self.E, key % self.E, RESIZE_EVICT, s, key))
                self.map[key] = -1
                self.owner[s] = -1
                self.stamp[s] = 0
        movers = sorted(s for s in keep if s >= C_new)
        vacant = sorted(s for s in range(C_new) if self.owner[s] < 0)
        assert len(vacant) >= len(movers)
        for src, dst in zip(movers, vacant):
            key = int(self.owner[src])
            self.owner[dst] = key
            self.stamp[dst] = self.stamp[src]
            self.map[key] = dst
            self.owner[src] = -1
        self.owner = self.owner[:C_new].copy()
        self.stamp = self.stamp[:C_new].copy()
        self.C = C_new
        return events

    # -- prefill with full-layer double buffering --------------------------
    def prefill(self, l0: int, l1: int, chunks: int = 1) -> tuple[list[Event], np.ndarray]:
        """Layers l0 .. l1-1 through the two full-layer buffers, `chunks`
        times in a row (a long prompt runs as consecutive chunks, each a full
        pass over the layers; step i of the passes uses buffer i mod 2).

        Returns the PREFILL_EVICT events of carving the buffers and the slot
        table int64 [chunks * (l1 - l0), E]: the slot each expert is read from
        at each step (its buffer slot when streamed, its own slot when
        resident).
        """
        E, C = self.E, self.C
        if C < 2 * E:
            raise CapacityError(f"prefill needs two full-layer buffers ({2 * E} slots), the cache has {C}")
        buf0 = C - 2 * E
        events = []
        for s in range(buf0, C):
            key = int(self.owner[s])
            if key >= 0:
                events.append(Event(self.calls, key // E, key % E, PREFILL_EVICT, s, key))
                self.map[key] = -1
                self.owner[s] = -1
                self.stamp[s] = 0
        n = l1 - l0
        table = np.zeros((chunks * n, E), dtype=np.int64)
        for i in range(chunks * n):
            layer, b = l0 + i % n, i % 2
            for e in range(E):
                key = layer * E + e
                s = int(self.map[key])
                if s < 0:  # streamed into the buffer
                    s = buf0 + b * E + e
                    old = int(self.owner[s])
                    if old >= 0:
                        self.map[old] = -1
                    self.owner[s] = key
                    self.map[key] = s
                self.stamp[s] = np.uint64(self.g + e)
                table[i, e] = s
            self.g += E
        return events, table

    # -- prefill when two full-layer buffers do not fit ----------------------
    def prefill_on_demand(self, layer: int, ids: np.ndarray) -> tuple[list[Event], dict[int, int]]:
        """One layer of a prefill whose cache cannot give two full-layer
        buffers (C < 2E): the layer's distinct routed experts, ascending, are
        accessed in consecutive chunks of at most C, each chunk exactly like
        one decode call (hits refresh recency, misses take victims by the
        usual rule and are loaded); the chunk's experts are evaluated before
        the next chunk may evict them.  Returns the events and the slot every
        expert of the layer was read from.
        """
        U = sorted(set(int(e) for e in np.asarray(ids).reshape(-1)))
        if self.C < 1 and U:
            raise CapacityError("prefill needs at least one slot")
        events, slot_of = [], {}
        for c0 in range(0, len(U), max(1, self.C)):
            chunk = np.array(U[c0:c0 + self.C], dtype=np.int64).reshape(1, -1)
            ev, slots = self.access(layer, chunk)
            events += ev
            for e, s in zip(chunk.reshape(-1), slots.reshape(-1)):
                slot_of[int(e)] = int(s)
        return events, slot_of

    def resident_keys(self) -> set[int]:
        return {int(k) for k in self.owner if k >= 0}


def hit_rate(events: list[Event]) -> float:
    """hits / (hits + misses) over distinct (call, layer, expert) accesses."""
    h = sum(1 for e in events if e.kind == HIT)
    m = sum(1 for e in events if e.kind == MISS)
    return h / (h + m) if h + m else float("nan")
