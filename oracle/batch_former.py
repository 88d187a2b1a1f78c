"""The batch former's oracle: TEST INFRASTRUCTURE ONLY.

Plain Python, written from the pages' description of the adapter-aware scheduler; it shares
no code with the library (``adapter_serving_gb300``) and never imports it.

``form_batch`` takes the pages' steps in their order:

* "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A: Batching Heterogeneous
  Adapters", "The adapter-aware scheduler": group the queue by adapter, visit the groups
  biggest first, take each whole while the batch has room (cut to fit), and stop admitting NEW
  adapters once the batch holds ``max_distinct`` of them and at least ``min_batch`` requests;
* the same section, "The fairness cost, which must be stated": a request older than the
  deadline is admitted regardless of grouping, and its adapter comes with it;
* the same page's revision R1 "The long tail needs a reserved batch slot": the oldest requests
  whose adapter has a group of size one get reserved places ahead of the grouping.

Readings where the pages leave a step open (listed in the design notes too): groups keep the
order of their first request and equal sizes keep that order; "oldest" means the longest wait
with ties in queue order; the age override runs first, then the tail slots, then the grouping;
an adapter admitted by an earlier step is not new to the grouping; the base-only group (-1) is
no adapter and never counts against the cap.
"""
from __future__ import annotations


def form_batch(queue_adapter, queue_waited_ms, max_batch, max_distinct, min_batch=1, tail_slots=0,
               max_queue_ms=0.0):
    """Returns (queue indices of the batch in batch order, number of distinct adapters >= 0)."""
    ids = [int(a) for a in queue_adapter]
    waited = [float(w) for w in queue_waited_ms]
    batch = []
    in_batch = set()
    adapters = set()

    def admit(i):
        batch.append(i)
        in_batch.add(i)
        if ids[i] >= 0:
            adapters.add(ids[i])

    def oldest_first(candidates):
        return sorted(candidates, key=lambda i: -waited[i])  # sorted() is stable: ties keep queue order

    # the age override: everything past the deadline, oldest first
    if max_queue_ms > 0:
        urgent = [i for i in range(len(ids)) if waited[i] > max_queue_ms]
        for i in oldest_first(urgent):
            if len(batch) == max_batch:
                break
            admit(i)

    # reserved tail slots: adapters with exactly one waiting request
    if tail_slots > 0:
        left = [i for i in range(len(ids)) if i not in in_batch]
        size = {}
        for i in left:
            size[ids[i]] = size.get(ids[i], 0) + 1
        singles = [i for i in left if ids[i] >= 0 and size[ids[i]] == 1]
        for i in oldest_first(singles)[:tail_slots]:
            if len(batch) == max_batch:
                break
            admit(i)

    # grouping, biggest groups first
    by_adapter = {}  # dicts keep insertion order: a group sits where its first request arrived
    for i in range(len(ids)):
        if i not in in_batch:
            by_adapter.setdefault(ids[i], []).append(i)
    order = sorted(by_adapter, key=lambda a: -len(by_adapter[a]))
    for a in order:
        if len(batch) >= max_batch:
            break
        new_adapter = a >= 0 and a not in adapters
        if new_adapter and len(adapters) >= max_distinct and len(batch) >= min_batch:
            continue
        for i in by_adapter[a][: max_batch - len(batch)]:
            admit(i)
    return batch, len(adapters)
