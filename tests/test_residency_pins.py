"""Pins for the residency-plan oracle (``oracle/residency.py``): worked
examples derived by hand from the rules of ``prepare_expert_jobs`` and
``pf_experts`` (cherenkov ``qwen4_exp`` engine, ``prefill/experts.rs``),
plus invariants and a brute-force check of the batch protocol: no fetch may
overwrite a slot that a batch it does not wait for still reads.
"""

import numpy as np
import pytest

from oracle import residency as R


def test_worked_example_first_chunk():
    # counts 3,0,5,1,5,2 over E = 6; an empty pool of 2 slots; ring 4,
    # group 2.  Ranking: experts 2 and 4 (5 rows, lower id first), 0 (3),
    # 5 (2), 3 (1): keep = {2, 4}, filled into slots 0 and 1.
    # Jobs in expert order: 0 ring slot 0 (record 2), 2 fill (record 0),
    # 3 ring slot 1 (record 3), 4 fill (record 1), 5 ring slot 2 (record 4).
    # Copies in that order, two per batch: batches 1,1,2,2,3; batch 3 waits
    # for batch 3 - 4/2 = 1.
    p = R.plan([3, 0, 5, 1, 5, 2], [-1, -1], [0, 0], call=1, ring=4, group=2)
    assert p["rec"] == [2, -1, 0, 3, 1, 4]
    assert p["batch"] == [1, -1, 1, 2, 2, 3]
    assert p["copies"] == [(0, 2), (2, 0), (3, 3), (4, 1), (5, 4)]
    assert p["n_batches"] == 4
    assert p["wait_for"] == [0, 0, 0, 1]
    assert p["pool_expert"] == [2, 4]
    assert p["pool_last"] == [1, 1]


def test_worked_example_second_chunk_evicts_only_unused_members():
    # Pool {2, 4} from the first chunk.  counts 4,6,0,0,1,0: keep = {1, 0}.
    # Expert 1: no free slot; slot 0 holds expert 2 (no rows now) -> evicted.
    # Expert 0: slot 1 holds expert 4, which has a row in this chunk, so it
    # stays and expert 0 streams (ring slot 0, record 2).  Expert 4 reads its
    # resident record in batch 0.
    p = R.plan([4, 6, 0, 0, 1, 0], [2, 4], [1, 1], call=2, ring=4, group=2)
    assert p["rec"] == [2, 0, -1, -1, 1, -1]
    assert p["batch"] == [1, 1, -1, -1, 0, -1]
    assert p["copies"] == [(0, 2), (1, 0)]
    assert p["n_batches"] == 2
    assert p["wait_for"] == [0, 0]
    assert p["pool_expert"] == [1, 4]
    assert p["pool_last"] == [2, 2]


def test_worked_example_least_recently_used_victim():
    # Pool of 3 holding experts 7, 8, 9, last used at calls 5, 3, 3; only
    # expert 0 has rows.  All three members are unused now; the oldest are
    # slots 1 and 2 (call 3), and the lower slot goes first.
    counts = [2] + [0] * 9
    p = R.plan(counts, [7, 8, 9], [5, 3, 3], call=6, ring=2, group=2)
    assert p["pool_expert"] == [7, 0, 9]
    assert p["pool_last"] == [5, 6, 3]
    assert p["rec"][0] == 1 and p["batch"][0] == 1
    assert p["copies"] == [(0, 1)]


def test_single_slot_pool_keeps_the_lower_id_on_a_tie():
    p = R.plan([3, 0, 5, 1, 5, 2], [-1], [0], call=1, ring=2, group=1)
    assert p["pool_expert"] == [2]
    # every other expert streams: 0, 3, 4, 5 take ring slots 0, 1, 0, 1
    assert p["rec"] == [1, -1, 0, 2, 1, 2]
    assert p["copies"] == [(0, 1), (2, 0), (3, 2), (4, 1), (5, 2)]
    assert p["batch"] == [1, -1, 2, 3, 4, 5]
    assert p["wait_for"] == [0, 0, 0, 1, 2, 3]


def test_ring_must_be_a_multiple_of_the_group():
    with pytest.raises(ValueError):
        R.plan([1, 1], [], [], call=1, ring=3, group=2)
    with pytest.raises(ValueError):
        R.plan([1, 1], [], [], call=1, ring=1, group=2)


def _check_protocol(counts, before, p, P, ring, group):
    """Invariants of one plan and a brute-force hazard check."""
    E = len(counts)
    active = [e for e in range(E) if counts[e] > 0]
    # one record per active expert, none for the rest
    for e in range(E):
        if counts[e] > 0:
            assert 0 <= p["rec"][e] < P + ring and p["batch"][e] >= 0
        else:
            assert p["rec"][e] == -1 and p["batch"][e] == -1
    # resident jobs are exactly the active experts that were members and stay
    members_before = {e for e in before if e >= 0}
    for e in active:
        resident = p["batch"][e] == 0
        assert resident == (e in members_before and e in p["pool_expert"])
        if p["rec"][e] < P:
            assert p["pool_expert"][p["rec"][e]] == e
    # members are distinct; a member evicted in this chunk had no rows
    after = [e for e in p["pool_expert"] if e >= 0]
    assert len(after) == len(set(after))
    for e in members_before - set(after):
        assert counts[e] == 0
    # copies: in ascending expert order, group per batch
    ex = [e for e, _ in p["copies"]]
    assert ex == sorted(ex)
    assert [p["batch"][e] for e in ex] == [1 + i // group for i in range(len(ex))]
    assert p["n_batches"] == 1 + -(-len(ex) // group)
    # the keep set is resident whenever enough slots could be freed
    by_use = sorted(active, key=lambda e: -counts[e])
    keep = by_use[:P]
    freeable = sum(1 for e in before if e < 0 or counts[e] == 0)
    new = [e for e in keep if e not in members_before]
    if len(new) <= freeable:
        assert set(keep) <= set(after)
    # hazards: batches run 0, 1, 2, ... on the GPU; fetch batch b starts once
    # batch wait_for[b] is done (so every batch <= wait_for[b] is done) and
    # may overlap any later batch.  No batch it may overlap reads a slot it
    # writes, and no two jobs of one batch write the same slot.
    readers = {}
    for e in active:
        readers.setdefault(p["rec"][e], []).append(p["batch"][e])
    for b in range(1, p["n_batches"]):
        written = [s for (e, s) in p["copies"] if p["batch"][e] == b]
        assert len(written) == len(set(written))
        for s in written:
            for rb in readers[s]:
                if rb >= b:
                    continue  # batch b itself, or a later batch that refetches the slot
                # an earlier reader of the slot must be done before the fetch
                assert rb <= p["wait_for"][b], (b, s, rb)


@pytest.mark.parametrize("seed", range(40))
def test_random_plans_meet_the_invariants(seed):
    rng = np.random.default_rng([seed, 901])
    E = int(rng.integers(1, 40))
    P = int(rng.integers(0, E + 3))
    group = int(rng.integers(1, 6))
    ring = group * int(rng.integers(1, 4))
    pool = [-1] * P
    last = [0] * P
    for call in range(1, 6):
        # skewed counts with many zeros
        counts = (rng.random(E) < 0.6) * rng.zipf(1.6, E).clip(max=50)
        before = list(pool)
        p = R.plan(counts, pool, last, call=call, ring=ring, group=group)
        _check_protocol(list(counts), before, p, P, ring, group)
        pool, last = p["pool_expert"], p["pool_last"]


def test_pool_as_large_as_the_expert_count_stops_streaming():
    counts = [3, 1, 4, 1, 5]
    p = R.plan(counts, [-1] * 5, [0] * 5, call=1, ring=2, group=2)
    assert sorted(e for e in p["pool_expert"] if e >= 0) == [0, 1, 2, 3, 4]
    p2 = R.plan(counts, p["pool_expert"], p["pool_last"], call=2, ring=2, group=2)
    assert p2["copies"] == [] and p2["n_batches"] == 1
    assert all(b == 0 for b in p2["batch"])


def test_empty_pool_streams_every_active_expert_in_order():
    counts = [0, 2, 0, 7, 1]
    p = R.plan(counts, [], [], call=1, ring=2, group=1)
    assert p["copies"] == [(1, 0), (3, 1), (4, 0)]
    assert p["wait_for"] == [0, 0, 0, 1]
