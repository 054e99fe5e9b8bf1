"""CPU oracle of the expert residency plan: which routed expert records stay
resident in device memory across chunks and which stream through a ring of
slots, in what batches, with which waits.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/`` use it.  It shares no code with the
CUDA library.

What it restates (cherenkov ``qwen4_exp`` engine, rustdoc source pages):

* ``prefill.rs`` module doc: records stream through a ring of pool slots; a
  fetch side fills batches ahead of the GPU, with two events per batch.
  ``RING`` slots, ``GROUP`` experts per fetch batch.
* ``prefill/experts.rs``, ``prepare_expert_jobs``: the experts with rows
  are ranked by their row count (descending; a stable sort of the
  ascending ids, so equal counts keep the lower id first); the first
  ``budget`` of them form the keep set.  Jobs follow in ascending expert
  order.  An expert that is kept, or whose record is already a member of
  the residency set, reads its record from the pool (acquiring a pool slot
  first when it is not yet resident, which fetches it); every other expert
  takes the next ring slot, ``ring_pos % RING``.
* ``prefill/experts.rs``, ``pf_experts``: the jobs go in batches of
  ``GROUP``.  Before the fetch side overwrites the ring slots of batch
  ``bi`` it waits until the GPU has finished batch ``bi - RING / GROUP``;
  after the fetch it signals "batch fetched", which the GPU waits for
  before it runs the batch.

Readings where the pages are silent or where this build departs:

* pool eviction (the body of ``res.acquire`` is not printed): a kept expert
  that is not resident takes the lowest free pool slot, else the slot of
  the least recently used member (lowest slot on ties) whose expert has no
  rows in this chunk.  With no such slot it streams through the ring for
  this chunk.  Members are never evicted for a chunk that uses them.
* batches hold only the jobs that copy a record (pool fills and ring
  jobs), ``GROUP`` at a time in ascending expert order; the jobs whose
  record is already resident, and the shared expert, form batch 0, which
  needs no fetch and runs first.
* a ring slot is reused only ``RING / GROUP`` batches later, so ``RING``
  must be a positive multiple of ``GROUP``.
"""

from __future__ import annotations

import numpy as np


def plan(counts, pool_expert, pool_last, call, ring, group):
    """One chunk's residency plan.

    counts       int [E]: rows routed to each expert in this chunk
    pool_expert  int [P]: expert held by each pool slot, -1 for a free slot
    pool_last    int [P]: call number of each slot's last use
    call         this chunk's call number (larger than every earlier one)
    ring, group  ring slots and copy jobs per fetch batch

    Returns a dict with the new pool state and the plan:
      rec[e]      record slot of expert e (pool slot, or P + ring slot; -1
                  when e has no rows)
      batch[e]    0 when e's record is resident, b >= 1 for the fetch batch
                  that copies it, -1 when e has no rows
      copies      list of (expert, record slot) in copy order
      n_batches   1 + number of fetch batches
      wait_for[b] the batch whose completion fetch batch b waits for before
                  it overwrites ring slots (0: none)
    """
    counts = np.asarray(counts, np.int64)
    E = counts.size
    pool_expert = [int(v) for v in pool_expert]
    pool_last = [int(v) for v in pool_last]
    P = len(pool_expert)
    if ring < group or group < 1 or ring % group:
        raise ValueError("ring must be a positive multiple of group")

    active = [e for e in range(E) if counts[e] > 0]
    # rank by row count, descending; Python's sort is stable, ids ascending
    by_use = sorted(active, key=lambda e: -counts[e])
    keep = by_use[:P]

    slot_of = {e: s for s, e in enumerate(pool_expert) if e >= 0}
    fills = {}  # expert -> pool slot it is copied into
    for e in keep:
        if e in slot_of:
            continue
        free = [s for s in range(P) if pool_expert[s] < 0]
        if free:
            s = free[0]
        else:
            victims = [s for s in range(P) if counts[pool_expert[s]] == 0]
            if not victims:
                continue  # streams through the ring this chunk
            s = min(victims, key=lambda v: (pool_last[v], v))
            del slot_of[pool_expert[s]]
        pool_expert[s] = e
        slot_of[e] = s
        fills[e] = s

    rec = [-1] * E
    batch = [-1] * E
    copies = []
    ring_pos = 0
    for e in active:
        if e in slot_of:
            s = slot_of[e]
            pool_last[s] = call
            rec[e] = s
            if e in fills:
                copies.append((e, s))
            else:
                batch[e] = 0
        else:
            rec[e] = P + ring_pos % ring
            ring_pos += 1
            copies.append((e, rec[e]))
    for i, (e, _) in enumerate(copies):
        batch[e] = 1 + i // group
    n_batches = 1 + (len(copies) + group - 1) // group
    lag = ring // group
    wait_for = [0] + [b - lag if b - lag >= 1 else 0 for b in range(1, n_batches)]
    return dict(rec=rec, batch=batch, copies=copies, n_batches=n_batches, wait_for=wait_for,
                pool_expert=pool_expert, pool_last=pool_last)


def miss_experts(p, pool_slots):
    """Experts of plan ``p`` whose record this chunk reads from a ring slot:
    the transient misses, which take the ``--miss-experts`` store
    (``prepare_expert_jobs``: only a resident pool record keeps the base
    layout)."""
    return {e for e, r in enumerate(p["rec"]) if r >= pool_slots}
