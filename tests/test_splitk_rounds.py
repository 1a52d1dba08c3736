"""CPU model of the tile kernel's split-K reduction through distributed shared memory.

The CTAs of a (1, 1, splitk) cluster each hold an FP32 partial tile; rank 0's pipeline
buffers hold `slots` partial tiles at once, so ranks 1 .. splitk - 1 hand theirs over in
rounds of `slots`: every thread of every CTA passes two cluster barriers per round; between
them the round's ranks write slot (rank - q0) of rank 0, and after the second rank 0 adds the
round's slots in rank order.  The model replays that schedule (the same round bounds as the
kernel) and checks that every partial is added exactly once, in rank order (the sum is
deterministic), that no slot is written while rank 0 may still read it, and that every rank
passes the same number of barriers (a cluster barrier must be reached by all CTAs).
"""
import itertools

import pytest


def rounds(splitk, slots):
    return (splitk - 1 + slots - 1) // slots if splitk > 1 else 0


def replay(splitk, slots):
    """Events of the schedule: ('write', round, rank, slot), ('add', round, rank, slot), barriers per rank."""
    events = []
    barriers = {r: 0 for r in range(splitk)}
    for rr in range(rounds(splitk, slots)):
        q0 = 1 + rr * slots
        q1 = min(q0 + slots, splitk)
        for r in range(splitk):       # first barrier: rank 0's slots are free
            barriers[r] += 1
        for r in range(q0, q1):
            events.append(("write", rr, r, r - q0))
        for r in range(splitk):       # second barrier: the round's partials have landed
            barriers[r] += 1
        for q in range(q0, q1):
            events.append(("add", rr, q, q - q0))
    return events, barriers


@pytest.mark.parametrize("splitk,slots", list(itertools.product(range(1, 9), range(1, 7))))
def test_every_partial_added_once_in_rank_order(splitk, slots):
    events, barriers = replay(splitk, slots)
    adds = [e for e in events if e[0] == "add"]
    assert [e[2] for e in adds] == list(range(1, splitk))           # ranks 1 .. splitk - 1, in order
    writes = {(e[1], e[2]): e[3] for e in events if e[0] == "write"}
    for _, rr, rank, slot in adds:
        assert writes[(rr, rank)] == slot and 0 <= slot < slots        # read from the slot that rank wrote
    # a slot is written in round rr only after rank 0 added round rr - 1 (the barrier between)
    for rr in range(1, rounds(splitk, slots)):
        last_add_prev = max(i for i, e in enumerate(events) if e[0] == "add" and e[1] == rr - 1)
        first_write = min(i for i, e in enumerate(events) if e[0] == "write" and e[1] == rr)
        assert last_add_prev < first_write
    assert len(set(barriers.values())) == 1                              # every rank, the same barrier count
    assert barriers[0] == 2 * rounds(splitk, slots)
    # one round when every partial fits at once (the plain two-barrier reduction)
    if splitk > 1 and splitk - 1 <= slots:
        assert rounds(splitk, slots) == 1


def test_sum_matches_a_plain_rank_ordered_sum():
    import numpy as np
    rng = np.random.default_rng(3)
    for splitk in range(2, 9):
        parts = [rng.standard_normal(64).astype(np.float32) for _ in range(splitk)]
        for slots in (1, 2, 3, 6):
            events, _ = replay(splitk, slots)
            acc = parts[0].copy()
            for e in events:
                if e[0] == "add":
                    acc = acc + parts[e[2]]
            want = parts[0].copy()
            for r in range(1, splitk):
                want = want + parts[r]
            assert np.array_equal(acc, want)      # bit-identical: the order does not depend on slots
