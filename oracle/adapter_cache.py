"""The adapter cache's oracle: TEST INFRASTRUCTURE ONLY.

Plain Python, written from the pages; it shares no code with the library and never imports it.

* "m07 -- Multi-Adapter (LoRA) Serving", section 7 "Deep Dive B: The Cold-Start Long Tail",
  "Eviction, and the trap in it": an adapter's value is its requests in the last hour divided by
  the bytes it holds; evict the lowest value first; never evict an adapter with in-flight
  requests (reference counted); while pinned bytes exceed a share of the budget, admit no new
  adapters (the pinning guard).
* the same page, revision R3 "The pinning guard was inconsistent": size the cache by Little's
  law -- pinned adapters = arrival rate of distinct adapters x mean generation time, budget
  = 2 x that x adapter size -- and put the guard at 80%.

Readings where the pages leave a step open (listed in the design notes too): "the last hour" is
a sliding window (requests with time > now - window count); equal values go to the adapter whose
latest request is older, then to the smaller id; eviction happens only to make room for a new
adapter; a request that cannot be placed even after evicting every unreferenced adapter changes
nothing.
"""
from __future__ import annotations

from fractions import Fraction


class AdapterCache:
    def __init__(self, budget_bytes, guard_fraction=0.8, window_s=3600.0):
        self.budget = int(budget_bytes)
        self.guard = float(guard_fraction)
        self.window = float(window_s)
        self.bytes = {}       # adapter -> bytes it holds while resident
        self.resident = set()
        self.ref = {}         # adapter -> in-flight sequences
        self.requests = {}    # adapter -> request times (all of them)
        self.clock = float("-inf")

    def _value(self, a, now):
        recent = [t for t in self.requests.get(a, []) if t > now - self.window]
        return Fraction(len(recent), self.bytes[a])

    def pinned_bytes(self):
        return sum(self.bytes[a] for a in self.resident if self.ref.get(a, 0) > 0)

    def used_bytes(self):
        return sum(self.bytes[a] for a in self.resident)

    def acquire(self, a, nbytes, now):
        """Returns ("ok", evicted, must_load) or ("pinned", [], False) or ("nomem", [], False)."""
        assert now >= self.clock, "request times never go back"
        self.clock = now
        if a in self.resident:
            assert self.bytes[a] == nbytes
            self.requests.setdefault(a, []).append(now)
            self.ref[a] = self.ref.get(a, 0) + 1
            return "ok", [], False
        if self.pinned_bytes() > self.guard * self.budget:
            return "pinned", [], False
        if nbytes > self.budget:
            return "nomem", [], False
        free = self.budget - self.used_bytes()
        unreferenced = [b for b in self.resident if self.ref.get(b, 0) == 0]
        latest = {b: max(self.requests.get(b, [float("-inf")])) for b in unreferenced}
        order = sorted(unreferenced, key=lambda b: (self._value(b, now), latest[b], b))
        evicted = []
        for b in order:
            if free >= nbytes:
                break
            evicted.append(b)
            free += self.bytes[b]
        if free < nbytes:
            return "nomem", [], False
        for b in evicted:
            self.resident.discard(b)
        self.bytes[a] = nbytes
        self.resident.add(a)
        self.ref[a] = 1
        self.requests.setdefault(a, []).append(now)
        return "ok", evicted, True

    def release(self, a):
        assert a in self.resident and self.ref.get(a, 0) > 0
        self.ref[a] -= 1


def little_pinned_adapters(distinct_arrivals_per_s, mean_generation_s):
    """Adapters pinned in steady state: arrival rate of distinct adapters x mean duration (R3)."""
    return distinct_arrivals_per_s * mean_generation_s


def little_cache_bytes(distinct_arrivals_per_s, mean_generation_s, adapter_bytes, headroom=2.0):
    """R3's sizing: headroom x pinned adapters x adapter size."""
    return headroom * little_pinned_adapters(distinct_arrivals_per_s, mean_generation_s) * adapter_bytes
