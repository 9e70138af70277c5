"""Host model of the work-item ring the persistent CTAs use to hand each
claimed item (index and geometry) from the producer thread to the CTA's
other roles (csrc/sched.cuh: ring_acquire / ring_publish / ring_wait /
ring_release over kRingSlots slots, each guarded by a "full" and an "empty"
mbarrier).

The model restates the ring's phase arithmetic against a model of the
mbarrier: a barrier counts arrivals of its current phase, completes the
phase when the count is reached, and a wait for parity P succeeds once the
current (incomplete) phase's parity differs from P, i.e. the phase with
parity P has completed.  Random interleavings of one producer and several
consumers (one of which keeps its slot for a while, as the forward's softmax
warps keep theirs until their epilogue) must deliver every round's item to
every consumer, in order, never a stale or overwritten one, and never
deadlock."""
from __future__ import annotations

import random

import pytest

SLOTS = 4  # kRingSlots


class MBarrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0  # index of the current, incomplete phase

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def test_parity(self, parity):
        return (self.phase & 1) != parity


def run(n_rounds, n_consumers, hold_max, seed):
    rng = random.Random(seed)
    full = [MBarrier(1) for _ in range(SLOTS)]
    empty = [MBarrier(n_consumers) for _ in range(SLOTS)]
    slot = [None] * SLOTS
    # the producer: round r -> acquire (wait empty), publish (write, arrive full)
    prod = {"r": 0}
    # consumer c: round r -> wait full, read, hold `hold` scheduler ticks, release
    cons = [{"r": 0, "state": "wait", "hold": 0, "seen": []} for _ in range(n_consumers)]
    ticks = 0
    while prod["r"] < n_rounds or any(c["r"] < n_rounds for c in cons):
        ticks += 1
        assert ticks < 200000, "deadlock"
        actors = []
        if prod["r"] < n_rounds:
            actors.append(("p", None))
        actors += [("c", i) for i, c in enumerate(cons) if c["r"] < n_rounds]
        kind, i = rng.choice(actors)
        if kind == "p":
            r = prod["r"]
            s, use = r % SLOTS, r // SLOTS
            if use > 0 and not empty[s].test_parity((use - 1) & 1):
                continue  # ring_acquire: slot still held
            slot[s] = ("item", r)
            full[s].arrive()  # ring_publish
            prod["r"] += 1
            continue
        c = cons[i]
        r = c["r"]
        s = r % SLOTS
        if c["state"] == "wait":
            if not full[s].test_parity((r // SLOTS) & 1):
                continue  # ring_wait: not published yet
            assert slot[s] == ("item", r), (i, r, slot[s])  # never stale, never overwritten
            c["seen"].append(r)
            c["state"] = "hold"
            c["hold"] = rng.randint(0, hold_max) if i == 0 else 0
        elif c["hold"] > 0:
            # the consumer still reads the slot: it must still hold round r's item
            assert slot[s] == ("item", r), (i, r, slot[s])
            c["hold"] -= 1
        else:
            empty[s].arrive()  # ring_release
            c["r"] += 1
            c["state"] = "wait"
    for c in cons:
        assert c["seen"] == list(range(n_rounds))


@pytest.mark.parametrize("seed", range(20))
def test_ring_delivers_every_item_in_order(seed):
    run(n_rounds=61, n_consumers=3, hold_max=40, seed=seed)


def test_ring_parity_would_alias_without_the_empty_wait():
    """The empty-barrier wait is what keeps the producer within SLOTS rounds
    of the slowest consumer: without it a consumer could read a slot two
    phases ahead of the one it waits for (parity aliasing)."""
    full = MBarrier(1)
    for _ in range(2):
        full.arrive()  # two publications into one slot with nobody reading
    # a consumer of the first publication (phase 0, parity 0) sees phase 2,
    # whose parity is 0 again: its wait does not succeed, it would wait for a
    # third publication -- the hazard the empty barrier rules out
    assert not full.test_parity(0)
