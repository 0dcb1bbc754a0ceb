"""Brute-force re-derivation of the slot cache, used only to pin the oracle.

It keeps no recency stamps and no LRU list.  Every decision is recomputed
from the full history: a slot's last touch is found by scanning the event log
backwards, an expert's demand count and last demand by scanning the log of
admissions.  It is slow (quadratic in the history) and meant for tiny pools.

Semantics (the same definition the oracle implements with a linked list):
one clock per pool, advanced once per admission; victims are the unpinned
slots not touched by the current admission, oldest last touch first, lowest
slot index on ties, never-touched (empty) slots first; misses are admitted in
ascending expert id up to the fetch cap; a prefetch does not advance the clock
and is refused by the LFRU guard as described in llama.cpp fork PR #126
("cuda : MoE look-ahead expert prefetch (PR-A consumer) + LFRU eviction
guard", section Eviction guard).
"""
from __future__ import annotations

FIELDS = (
    "calls", "lookups", "hits", "misses", "fetched", "overflow_routes", "evictions",
    "invalid_routes", "pf_requests", "pf_invalid", "pf_resident", "pf_filled",
    "pf_dropped_guard", "pf_no_victim", "pf_evictions", "status_bits",
)


class Brute:
    def __init__(self, L: int, E: int, S: int, per_layer: bool = False):
        self.L, self.E, self.S = L, E, S
        self.per_layer = per_layer
        self.P = L if per_layer else 1
        self.slot_key = [[-1] * S for _ in range(self.P)]
        self.pinned = [[False] * S for _ in range(self.P)]
        self.log = [[] for _ in range(self.P)]      # (time, slot, kind)
        self.time = [1] * self.P
        self.demand_log: list[tuple[int, set]] = []  # (time, keys) per admission
        self.decode_freq = [0] * (L * E)
        self.stats = [{f: 0 for f in FIELDS} for _ in range(L)]

    def pool(self, layer: int) -> int:
        return layer if self.per_layer else 0

    def key(self, layer: int, e: int) -> int:
        return layer * self.E + e

    def last_touch(self, p: int, s: int) -> int:
        for t, slot, kind in reversed(self.log[p]):
            if slot == s:
                return t if kind == "touch" else 0
        return 0

    def resident(self, p: int, key: int) -> int:
        for s, k in enumerate(self.slot_key[p]):
            if k == key:
                return s
        return -1

    def eligible(self, p: int) -> list[int]:
        t = self.time[p]
        el = [s for s in range(self.S)
              if not self.pinned[p][s] and self.last_touch(p, s) < t]
        return sorted(el, key=lambda s: (self.last_touch(p, s), s))

    def prefill(self, layer: int, ids) -> None:
        p = self.pool(layer)
        for e in ids:
            s = self.slot_key[p].index(-1)
            self.slot_key[p][s] = self.key(layer, e)
            self.log[p].append((self.time[p], s, "touch"))

    def pin(self, layer: int, slot: int, pinned: bool) -> None:
        self.pinned[self.pool(layer)][slot] = bool(pinned)

    def admit(self, layer: int, ids, cap: int = -1) -> dict:
        p = self.pool(layer)
        st = self.stats[layer]
        self.time[p] += 1
        t = self.time[p]
        st["calls"] += 1
        valid = [0 <= e < self.E for e in ids]
        for v in valid:
            if not v:
                st["invalid_routes"] += 1
                st["status_bits"] |= 1
        D = sorted({e for e, v in zip(ids, valid) if v})
        for e, v in zip(ids, valid):
            if v:
                self.decode_freq[self.key(layer, e)] += 1
        st["lookups"] += len(D)
        self.demand_log.append((t, {self.key(layer, e) for e in D}))
        M = []
        for e in D:
            s = self.resident(p, self.key(layer, e))
            if s >= 0:
                self.log[p].append((t, s, "touch"))
                st["hits"] += 1
            else:
                M.append(e)
        st["misses"] += len(M)
        A = M if cap < 0 else M[:cap]
        el = self.eligible(p)
        if len(el) < len(A):
            A = A[:len(el)]
            st["status_bits"] |= 2
        plan = []
        for e, s in zip(A, el):
            if self.slot_key[p][s] >= 0:
                st["evictions"] += 1
            self.slot_key[p][s] = self.key(layer, e)
            self.log[p].append((t, s, "touch"))
            plan.append((s, layer, e))
            st["fetched"] += 1
        slots = []
        for e, v in zip(ids, valid):
            if not v:
                slots.append(-1)
                continue
            s = self.resident(p, self.key(layer, e))
            slots.append(s)
            if s < 0:
                st["overflow_routes"] += 1
        groups = []
        for e in D:
            s = self.resident(p, self.key(layer, e))
            if s >= 0:
                groups.append((s, [r for r, (i, v) in enumerate(zip(ids, valid)) if v and i == e]))
        return {"slots": slots, "plan": plan, "groups": groups}

    def score(self, key: int, t: int) -> int:
        times = [tt for tt, keys in self.demand_log if key in keys]
        f = min(len(times), (1 << 24) - 1)
        rec = 0 if not times else 255 - min(255, t - max(times))
        return (f << 8) | rec

    def prefetch(self, layer: int, pred) -> list:
        p = self.pool(layer)
        st = self.stats[layer]
        t = self.time[p]
        for e in pred:
            if not 0 <= e < self.E:
                st["pf_invalid"] += 1
        P = sorted({e for e in pred if 0 <= e < self.E})
        st["pf_requests"] += len(P)
        plan = []
        for e in P:
            key = self.key(layer, e)
            if self.resident(p, key) >= 0:
                st["pf_resident"] += 1
                continue
            el = self.eligible(p)
            if not el:
                st["pf_no_victim"] += 1
                continue
            s = el[0]
            old = self.slot_key[p][s]
            if old >= 0:
                demands = sum(1 for _, keys in self.demand_log if old in keys)
                if demands >= 2 and 4 * self.score(old, t) > 5 * self.score(key, t) + 4 * (4 << 8):
                    st["pf_dropped_guard"] += 1
                    continue
                st["pf_evictions"] += 1
            self.slot_key[p][s] = key
            self.log[p].append((t, s, "touch"))
            plan.append((s, layer, e))
            st["pf_filled"] += 1
        return plan

    def rollback(self, plan) -> None:
        for s, layer, e in plan:
            p = self.pool(layer)
            if self.slot_key[p][s] == self.key(layer, e):
                self.slot_key[p][s] = -1
                self.log[p].append((self.time[p], s, "empty"))
