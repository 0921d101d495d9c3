"""CPU model of the fold kernels' shared-memory ring protocol.

The kernels stream items (shrink k-chunks, then expand j-chunks) through `ns`
ring slots guarded by a full and an empty mbarrier per slot, and wait with
mbarrier parity tests. A parity test only tells the current phase of a barrier
from the one before it: if a waiter can be two phases ahead, the wait passes
falsely and a later arrival lands in the wrong phase. This model replays the
kernels' exact schedule (every producer warp serves every item in order and
arrives once per item; consumers either all take every item in order, or, for
shrink items, the KSG warps that own a slot (KSG = 1 or 2) take its items and
each releases it with 8 / KSG arrivals) under random interleavings and checks
that no parity wait passes early, no arrival lands in a wrong phase, and the
schedule never deadlocks, including across the two cluster barriers between
shrink and expand, and in the single-CTA form where the exchange barrier holds
only the consumer warps while the producer keeps issuing.
It also shows that a schedule in which producer warps split items by index
(the broken variant) fails.
"""
from __future__ import annotations

import random

import pytest

PRODUCER_WARPS, CONSUMER_WARPS = 4, 8


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phase, self.tx = count, count, 0, 0

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, phase, tx=0):
        assert phase == self.phase, f"arrival for phase {phase} lands in phase {self.phase}"
        self.tx += tx
        self.pending -= 1
        self._check()

    def expect_tx(self, phase, tx):
        assert phase == self.phase, f"bytes for phase {phase} expected in phase {self.phase}"
        self.tx += tx

    def complete_tx(self, b):
        self.tx -= b
        self._check()

    def try_wait(self, phase):
        ok = (self.phase & 1) != (phase & 1)        # the hardware parity rule
        if ok:
            assert self.phase > phase, f"parity wait for phase {phase} passed in phase {self.phase}"
        return ok


def run(ns, n_shrink, n_items, slot_parallel, seed, producer_split="all", passes=None, ksg=1, cl1=False,
        full_release=False, late=False):
    """`passes`: [(n_shrink, n_items), ...] folded one after the other by one
    CTA; ring item numbers continue across passes and a CTA barrier separates them.
    ksg: warps per slot in slot-parallel shrinks (at most CONSUMER_WARPS // ns).
    cl1: single-CTA units: the producer issues every item without the exchange
    barriers, which only the consumer warps take.
    full_release: each owner warp releases a shrink slot with all eight arrivals
    (the broken variant when two warps own a slot).
    late: the late-wait order: before the exchange barriers the producer issues
    the shrink items and, with cluster peers, the first part (adapter rows, no
    arrival) of the expand items whose slots the shrink frees; after them it
    completes those items (out rows and its arrival), then the rest."""
    ksg = max(1, min(ksg, CONSUMER_WARPS // ns))
    rng = random.Random(seed)
    full = [Barrier(PRODUCER_WARPS) for _ in range(ns)]
    empty = [Barrier(CONSUMER_WARPS) for _ in range(ns)]
    passes = passes or [(n_shrink, n_items)]
    shrink_items = set()
    it0 = 0
    bounds = []
    for ps, pn in passes:
        bounds.append((it0, ps, pn))
        shrink_items.update(range(it0, it0 + ps))
        it0 += pn

    def producer(pw):
        prog = []
        for base, ps, pn in bounds:
            pre = ps if late else min(pn, ps + ns)
            early = min(pn, ps + ns) if (late and not cl1) else ps
            if producer_split == "all":
                a, b = list(range(pre)), list(range(max(pre, early), pn))
            else:   # items dealt to warps by index (broken)
                a = [i for i in range(pre) if i % PRODUCER_WARPS == pw]
                b = [i for i in range(pre, pn) if i % PRODUCER_WARPS == pw]
            first = [("W", base + i) for i in range(ps, early)]     # part 1: slot wait, adapter rows
            second = [("A", base + i) for i in range(ps, early)]    # part 2: out rows, arrival
            syncs = [] if cl1 else ["SYNC", "SYNC"]
            prog += [base + i for i in a] + first + syncs + second + [base + i for i in b] + ["SYNC"]
        return prog

    def consumer(w):
        prog = []
        for base, ps, pn in bounds:
            if slot_parallel:   # shrink items: the slot's owner warps; expand items: every warp in order
                sh = [base + i for i in range(ps) if (base + i) % ns == w % ns] if w < ns * ksg else []
            else:
                sh = [base + i for i in range(ps)]
            ex = ["CSYNC", "CSYNC"] if cl1 else ["SYNC", "SYNC"]
            prog += sh + ex + [base + i for i in range(ps, pn)] + ["SYNC"]
        return prog

    agents = [("P", producer(p)) for p in range(PRODUCER_WARPS)] + \
             [("C", consumer(w)) for w in range(CONSUMER_WARPS)]
    pc = [0] * len(agents)
    waited = [False] * len(agents)
    at_sync = [None] * len(agents)
    inflight = []
    per_copy = 1
    for _ in range(500000):
        live = [i for i in range(len(agents)) if pc[i] < len(agents[i][1])]
        if not live and not inflight:
            return
        choice = rng.choice(live + (["land"] if inflight else []))
        if choice == "land":
            s = inflight.pop(rng.randrange(len(inflight)))
            full[s].complete_tx(per_copy)
            continue
        kind, prog = agents[choice]
        op = prog[pc[choice]]
        if op in ("SYNC", "CSYNC"):
            # a barrier of every warp (SYNC) or of the consumer warps only (CSYNC)
            sid = (op, sum(1 for x in prog[:pc[choice] + 1] if x == op))
            at_sync[choice] = sid
            group = [i for i in range(len(agents)) if op == "SYNC" or agents[i][0] == "C"]
            if all(at_sync[i] == sid for i in group):
                for i in group:
                    pc[i] += 1
                    at_sync[i] = None
            continue
        part = None
        if isinstance(op, tuple):
            part, op = op
        s, u = op % ns, op // ns
        if kind == "P":
            if part != "A" and not waited[choice]:
                waited[choice] = u == 0 or empty[s].try_wait(u - 1)
                continue
            if part == "W":            # adapter rows: bytes in flight, no arrival yet
                full[s].expect_tx(u, per_copy)
            else:
                full[s].arrive(u, tx=per_copy)
            inflight.append(s)
        else:
            if not waited[choice]:
                waited[choice] = full[s].try_wait(u)
                continue
            n_arr = CONSUMER_WARPS if full_release else CONSUMER_WARPS // ksg
            for _ in range(n_arr if (slot_parallel and op in shrink_items) else 1):
                empty[s].arrive(u)
        waited[choice] = False
        pc[choice] += 1
    raise AssertionError("no progress: the schedule deadlocks")


@pytest.mark.parametrize("slot_parallel", [False, True])
@pytest.mark.parametrize("ns", [2, 3, 4, 6, 8])
def test_ring_schedule_is_sound(slot_parallel, ns):
    for n_shrink in (0, 1, 5, 16):
        for n_exp in (0, 1, 3, 32):
            for seed in range(3):
                run(ns, n_shrink, n_shrink + n_exp, slot_parallel, seed)


@pytest.mark.parametrize("slot_parallel", [False, True])
@pytest.mark.parametrize("ns", [2, 3, 5])
def test_ring_schedule_across_passes_is_sound(slot_parallel, ns):
    # item counts of successive passes leave the ring at every offset
    for passes in ([(1, 4), (2, 9), (1, 1)], [(3, 8), (0, 5), (4, 4), (2, 7)], [(5, 6)] * 4):
        for seed in range(3):
            run(ns, 0, 0, slot_parallel, seed, passes=passes)


@pytest.mark.parametrize("ns", [2, 3, 4, 5, 8])
def test_single_cta_units_with_two_warps_per_slot_are_sound(ns):
    """The MoE fold's schedule: slot-parallel shrinks with up to two warps per
    slot, the exchange barrier of the consumer warps only, passes one after the
    other."""
    for passes in ([(4, 16)], [(5, 20), (1, 4), (3, 12)], [(0, 3), (6, 6)], [(2, 2)] * 3):
        for seed in range(3):
            run(ns, 0, 0, True, seed, passes=passes, ksg=2, cl1=True)
            run(ns, 0, 0, False, seed, passes=passes, ksg=1, cl1=True)


def test_two_owner_warps_releasing_a_slot_in_full_is_unsound():
    failures = 0
    for seed in range(10):
        try:
            run(4, 0, 0, True, seed, passes=[(8, 20)], ksg=2, cl1=True, full_release=True)
        except AssertionError:
            failures += 1
    assert failures == 10


def test_items_split_by_index_across_producers_is_unsound():
    failures = 0
    for seed in range(20):
        try:
            run(2, 12, 16, False, seed, producer_split="by_index")
        except AssertionError:
            failures += 1
    assert failures == 20


@pytest.mark.parametrize("slot_parallel", [False, True])
@pytest.mark.parametrize("ns", [2, 3, 4, 8])
def test_late_wait_order_is_sound(slot_parallel, ns):
    """Inputs-ready launches: the producer holds every expand item back until
    after the exchange barriers (cluster units) or issues in item order (single
    CTA units); both still complete for every item count and pass sequence."""
    for passes in ([(1, 4)], [(5, 9), (0, 3)], [(16, 48)], [(3, 3), (2, 7)]):
        for seed in range(3):
            run(ns, 0, 0, slot_parallel, seed, passes=passes, late=True)
            run(ns, 0, 0, slot_parallel, seed, passes=passes, late=True, cl1=True,
                ksg=2 if slot_parallel else 1)
