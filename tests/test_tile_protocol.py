"""The tensor-core tile kernel's synchronisation protocol, checked on the CPU.

csrc/q4_tc.cu runs, per CTA: an X producer (one TMA tile per 64-wide group into SX
stages), a code producer (one TMA stage of 4 groups into SW stages, freed by both
decode teams), two decode teams (team t takes groups 4ws + t and 4ws + t + 2 of code
stage ws, writes the group's A operand into one of SA stages and then waits for
its X tile), one MMA issuer that meets the decode team (and, in the exact form, the
accumulate warps) on a ring of kRing named barriers before issuing a group's MMAs,
and one tcgen05.commit per group into a ring of kRing mbarriers.  In the exact form
the accumulate warps read each group's accumulator buffer (NB of them) and hand it
back through the issue barrier of group i + NB; in the folded form there is one
accumulator and they wait for the last commit only.

This model replays that protocol with mbarrier parity semantics (a wait for phase
k passes once k + 1 phases completed, and cannot tell k + 2 from k), copies that
land at any time, MMAs that complete in issue order at any time, and roles at any
relative speed.  It checks that no stage is overwritten while in use, no MMA runs
before its operands are in place, no waiter falls two phases behind, no arrival
lands on a named barrier still in use for an earlier group, and that the run
always completes.  Shrinking the barrier rings below the stage rings (a rule the
kernel's static_asserts keep) makes the model find violations.
"""
import random

import pytest

K_RING = 8
GROUPS_PER_STAGE = 4
# token-tile width -> (SX, SA, NB, SW) of the exact form; the folded form has NB = 1 and,
# at 256, six X stages
CFG = {256: (4, 4, 2, 2), 128: (8, 8, 2, 4), 64: (8, 8, 4, 4), 32: (8, 8, 8, 4), 16: (8, 8, 8, 4)}


class Violation(Exception):
    pass


def replay(ng, sx, sa, nb, sw, fold, rng, k_ring=K_RING, acc_in_barrier=True, max_steps=200000):
    nws = -(-ng // GROUPS_PER_STAGE)
    mma_done = [0] * k_ring                    # completed phases per commit barrier
    x_full, c_full = [0] * sx, [0] * sw
    c_empty, c_empty_arr = [0] * sw, [0] * sw
    nbar_gen = [0] * k_ring                    # completed generations per named barrier
    nbar_arr = [set() for _ in range(k_ring)]
    need = {"team", "issuer"} | (set() if fold or not acc_in_barrier else {"acc"})
    x_landed, a_written, c_read = set(), set(), {}
    x_inflight, c_inflight, mma_queue = [], [], []
    mma_completed = 0
    d_read = set()

    def wait_ok(count, phase, who):
        if count >= phase + 2:
            raise Violation(f"{who} two phases behind")
        return count > phase

    def arrive(group, who):
        j = group % k_ring
        if nbar_gen[j] != group // k_ring:
            raise Violation(f"{who} arrived for group {group} on barrier {j} still in use")
        role = "team" if who.startswith("team") else who
        if role in nbar_arr[j]:
            raise Violation(f"{who} arrived twice for group {group}")
        nbar_arr[j].add(role)

    # program counters
    px = 0
    pc = 0
    teams = [{"ws": 0, "h": -1, "step": "wait_c"} for _ in range(2)]
    pi = 0
    acc = {"i": 0, "pre": 0, "step": "pre"} if not fold else {"done": False}

    def team_groups(t, ws):
        return [i for i in (ws * 4 + t, ws * 4 + t + 2) if i < ng]

    for _ in range(max_steps):
        acts = []
        # X producer
        if px < ng:
            i = px
            if i < sx or wait_ok(mma_done[(i - sx) % k_ring], (i - sx) // k_ring, "X producer"):
                acts.append("x_issue")
        if x_inflight:
            acts.append("x_land")
        # code producer
        if pc < nws:
            ws = pc
            if wait_ok(c_empty[ws % sw] + 1, ws // sw, "code producer"):   # first use passes at once
                acts.append("c_issue")
        if c_inflight:
            acts.append("c_land")
        # decode teams
        for t in range(2):
            st = teams[t]
            if st["ws"] < nws:
                acts.append(("team", t))
        # issuer
        if pi < ng:
            j = pi % k_ring
            if nbar_gen[j] == pi // k_ring and need <= nbar_arr[j] | {"issuer"}:
                acts.append("issue")
        if mma_queue:
            acts.append("mma_done")
        # accumulate warps
        if not fold and acc["i"] < ng:
            acts.append("acc")
        if not acts:
            break
        a = rng.choice(acts)
        if a == "x_issue":
            i = px
            if i >= sx and mma_completed <= i - sx:
                raise Violation(f"X stage {i % sx} overwritten before MMA {i - sx} finished")
            if x_full[i % sx] != i // sx:
                raise Violation(f"X barrier {i % sx} rearmed early")
            x_inflight.append(i)
            px += 1
        elif a == "x_land":
            i = x_inflight.pop(rng.randrange(len(x_inflight)))
            x_full[i % sx] += 1
            x_landed.add(i)
        elif a == "c_issue":
            ws = pc
            if ws >= sw and c_read.get(ws - sw, 0) < 2:
                raise Violation(f"code stage {ws % sw} refilled before both teams read it")
            c_inflight.append(ws)
            pc += 1
        elif a == "c_land":
            ws = c_inflight.pop(rng.randrange(len(c_inflight)))
            c_full[ws % sw] += 1
        elif a == "issue":
            i = pi
            if i not in a_written or i not in x_landed:
                raise Violation(f"MMA {i} issued before its operands were in place")
            if not fold and i >= nb and (i - nb) not in d_read:
                raise Violation(f"MMA {i} overwrites buffer {i % nb} before group {i - nb} was read")
            j = i % k_ring
            nbar_gen[j] += 1
            nbar_arr[j] = set()
            mma_queue.append(i)
            pi += 1
        elif a == "mma_done":
            i = mma_queue.pop(0)
            mma_completed += 1
            mma_done[i % k_ring] += 1
        elif a == "acc":
            if acc["step"] == "pre":
                # the first NB groups find their buffers free
                if acc["pre"] < min(nb, ng):
                    if acc_in_barrier:
                        arrive(acc["pre"], "acc")
                    acc["pre"] += 1
                if acc["pre"] >= min(nb, ng):
                    acc["step"] = "wait"
            else:
                i = acc["i"]
                if wait_ok(mma_done[i % k_ring], i // k_ring, "accumulate warps"):
                    d_read.add(i)
                    if i + nb < ng and acc_in_barrier:
                        arrive(i + nb, "acc")
                    acc["i"] += 1
        else:
            t = a[1]
            st = teams[t]
            ws = st["ws"]
            if st["step"] == "wait_c":
                if wait_ok(c_full[ws % sw], ws // sw, f"team {t}"):
                    c_read[ws] = c_read.get(ws, 0) + 1
                    c_empty_arr[ws % sw] += 1
                    if c_empty_arr[ws % sw] == 2:
                        c_empty_arr[ws % sw] = 0
                        c_empty[ws % sw] += 1
                    st["groups"] = team_groups(t, ws)
                    st["step"] = "wait_a"
            elif not st["groups"]:
                st["ws"] += 1
                st["step"] = "wait_c"
            else:
                i = st["groups"][0]
                if st["step"] == "wait_a":
                    if i < sa or wait_ok(mma_done[(i - sa) % k_ring], (i - sa) // k_ring, f"team {t}"):
                        if i >= sa and mma_completed <= i - sa:
                            raise Violation(f"A stage {i % sa} overwritten before MMA {i - sa} finished")
                        a_written.add(i)
                        st["step"] = "wait_x"
                elif st["step"] == "wait_x":
                    if wait_ok(x_full[i % sx], i // sx, f"team {t}"):
                        arrive(i, f"team {t}")
                        st["groups"].pop(0)
                        st["step"] = "wait_a"
    finished = (px == ng and pc == nws and pi == ng and not mma_queue and not x_inflight and not c_inflight
                and all(s["ws"] >= nws for s in teams) and (fold or acc["i"] >= ng))
    if not finished:
        raise Violation("deadlock: no role can make progress")
    return mma_completed


@pytest.mark.parametrize("bn", sorted(CFG))
@pytest.mark.parametrize("fold", [False, True])
def test_tile_protocol_is_safe(bn, fold):
    sx, sa, nb, sw = CFG[bn]
    if fold:
        nb = 1
        if bn == 256:
            sx = 6
    rng = random.Random(bn * 7 + fold)
    for ng in (1, 2, 3, 5, 8, 9, 17, 40):
        for _ in range(25):
            assert replay(ng, sx, sa, nb, sw, fold, rng) == ng


def test_model_finds_a_ring_shorter_than_the_stages():
    # a commit ring of 4 behind 8 X stages: the X producer (or a team) falls two phases behind
    rng = random.Random(1)
    found = False
    for _ in range(200):
        try:
            replay(40, 8, 8, 2, 4, False, rng, k_ring=4)
        except Violation:
            found = True
            break
    assert found


def test_model_finds_missing_buffer_handback():
    # the exact form with the accumulate warps left out of the issue barrier (the folded
    # form's barrier set): nothing stops MMA i + NB from overwriting a buffer not yet read
    rng = random.Random(2)
    found = False
    for _ in range(200):
        try:
            replay(20, 4, 4, 2, 2, False, rng, acc_in_barrier=False)
        except Violation:
            found = True
            break
    assert found
