"""The batch former's oracle: TEST INFRASTRUCTURE ONLY.

Plain Python, written from the pages' prose rules for the adapter-aware scheduler; it shares no
code with the library (``adapter_serving_gb300``) and never imports it.

The rules, from "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A: Batching
Heterogeneous Adapters":

* "The adapter-aware scheduler": requests of one adapter are batched together, bigger groups
  first, while the batch has room (a group that does not fit is cut); once the batch holds
  ``max_distinct`` adapters and at least ``min_batch`` requests, no NEW adapter is admitted;
* "The fairness cost, which must be stated": a request that has waited longer than the
  deadline is admitted regardless, and its adapter comes with it;
* revision R1 "The long tail needs a reserved batch slot": a few places are reserved for the
  oldest requests whose adapter has only that one request waiting.

This restatement decides admission request by request from explicit ranking keys, in three
phases with the readings named in the design notes (B-1..B-8):

1. overdue requests (wait > deadline), ranked by (longest wait, arrival), until the batch is
   full;
2. the remaining requests that are the only waiting request of their adapter (never the
   base-only id -1), ranked the same way, up to ``tail_slots`` of them and the batch's room;
3. everything else, ranked by (size of its adapter's remaining group descending, arrival of
   that group's first remaining request, arrival): a group is decided at its first request --
   refused if it brings a new adapter while the cap and MIN_BATCH are both reached -- and an
   admitted group's requests enter while the batch has room.

An adapter admitted in phases 1 or 2 is not new in phase 3; the base-only group is never an
adapter.
"""
from __future__ import annotations


def form_batch(queue_adapter, queue_waited_ms, max_batch, max_distinct, min_batch=1, tail_slots=0,
               max_queue_ms=0.0):
    """Returns (queue indices of the batch in batch order, number of distinct adapters >= 0)."""
    ids = [int(a) for a in queue_adapter]
    waited = [float(w) for w in queue_waited_ms]
    n = len(ids)

    def by_age(i):  # longest wait first; equal waits in arrival order
        return (-waited[i], i)

    chosen = []

    # phase 1: past the deadline
    if max_queue_ms > 0:
        overdue = sorted((i for i in range(n) if waited[i] > max_queue_ms), key=by_age)
        chosen += overdue[:max_batch]

    # phase 2: reserved places for adapters with a single waiting request
    taken = set(chosen)
    rest = [i for i in range(n) if i not in taken]
    count = {}
    for i in rest:
        count[ids[i]] = count.get(ids[i], 0) + 1
    lone = sorted((i for i in rest if ids[i] >= 0 and count[ids[i]] == 1), key=by_age)
    room = max_batch - len(chosen)
    chosen += lone[:max(0, min(tail_slots, room))]

    # phase 3: grouping
    taken = set(chosen)
    rest = [i for i in range(n) if i not in taken]
    size, first = {}, {}
    for i in rest:
        size[ids[i]] = size.get(ids[i], 0) + 1
        first.setdefault(ids[i], i)  # rest is in arrival order, so this is the earliest
    order = sorted(rest, key=lambda i: (-size[ids[i]], first[ids[i]], i))
    have = {ids[i] for i in chosen if ids[i] >= 0}
    verdict = {}  # adapter -> admitted or not, decided at its group's first request
    for i in order:
        if len(chosen) >= max_batch:
            break
        a = ids[i]
        if a not in verdict:
            brings_new = a >= 0 and a not in have
            verdict[a] = not (brings_new and len(have) >= max_distinct and len(chosen) >= min_batch)
            if verdict[a] and a >= 0:
                have.add(a)
        if verdict[a]:
            chosen.append(i)
    return chosen, len(have)
