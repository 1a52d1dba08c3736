"""The decode GEMV's shared-memory ring protocol, checked on the CPU.

The streaming kernel (csrc/q4_gemv.cu) has one producer that issues row blocks
in order into `slots` buffers, and W consumer warps that walk (block, column
group) items w, w + W, ...; a buffer is refilled only after all items of its
previous block arrived on its "slot free" barrier.  Consumers wait on "block
landed" mbarriers by phase parity, which cannot tell phase p from p - 2, so the
kernel keeps nfull = slots + lead such barriers (lead = the largest block step
between a warp's consecutive items).  This model replays the protocol with
mbarrier parity semantics, copies that land in any order, and warps at any
relative speed, and checks that no consumer ever reads a block before it landed,
that no barrier is rearmed while its previous block is in flight, and that the
run always completes.  With nfull = slots the same model finds violations.
"""
import random

import pytest


def lead_of(nj, nw):
    return nw // nj + (1 if nw % nj else 0)


def consumers_for(nj, max_consumers=15):
    whole = (max_consumers // nj) * nj if nj <= max_consumers else 0
    return whole if whole >= max_consumers - 3 else max_consumers


def replay(nj, nw, slots, nfull, nb, rng, max_steps=100000):
    full_done = [0] * nfull                  # completed phases per "block landed" barrier
    free_done = [0] * slots                  # completed phases per "slot free" barrier
    free_cnt = [0] * slots
    inflight, landed = set(), set()

    def issue(b):
        if full_done[b % nfull] != b // nfull:
            return f"barrier {b % nfull} rearmed for block {b} before block {b - nfull} landed"
        inflight.add(b)
        return None

    for b in range(min(nb, slots)):
        err = issue(b)
        if err:
            return err
    issued = min(nb, slots)
    items = nb * nj
    nxt = {w: w for w in range(nw)}
    for _ in range(max_steps):
        acts = []
        if inflight:
            acts.append(("land", None))
        if issued < nb:
            b = issued
            if (free_done[b % slots] & 1) != (((b // slots) & 1) ^ 1):
                acts.append(("issue", None))
        for w, it in nxt.items():
            if it < items:
                b = it // nj
                if (full_done[b % nfull] & 1) != ((b // nfull) & 1):
                    acts.append(("consume", w))
        if not acts:
            done = all(it >= items for it in nxt.values()) and issued == nb
            return None if done else "deadlock"
        kind, w = rng.choice(acts)
        if kind == "land":
            b = rng.choice(sorted(inflight))
            inflight.remove(b)
            landed.add(b)
            full_done[b % nfull] += 1
        elif kind == "issue":
            err = issue(issued)
            if err:
                return err
            issued += 1
        else:
            it = nxt[w]
            b = it // nj
            if b not in landed:
                return f"warp {w} passed the wait for block {b} before it landed"
            s = b % slots
            free_cnt[s] += 1
            if free_cnt[s] == nj:
                free_cnt[s] = 0
                free_done[s] += 1
            nxt[w] = it + nw
    return "no progress bound reached"


CASES = [(nj, slots, nb) for nj in (1, 2, 4, 5, 8, 17) for slots in (2, 3, 9) for nb in (5, 29)]


@pytest.mark.parametrize("nj,slots,nb", CASES)
def test_ring_with_lead_barriers_is_safe(nj, slots, nb):
    nw = consumers_for(nj)
    rng = random.Random(nj * 1000 + slots * 10 + nb)
    for _ in range(20):
        assert replay(nj, nw, slots, slots + lead_of(nj, nw), nb, rng) is None


def test_ring_without_lead_barriers_is_not_safe():
    # the model is sharp enough to see the hazard the extra barriers remove
    rng = random.Random(7)
    failures = sum(replay(4, 12, 5, 5, 29, rng) is not None for _ in range(20))
    assert failures > 0
