"""A model of the split-K decode kernel's stage ring, run on the CPU: one producer
issuing each slab's copy into stage i mod NS after the stage's previous round was
given back by every value group, and G groups of wpg consumer warps, warp w of a group
taking slabs w, w + wpg, ...  Barriers follow the mbarrier rules that matter here: a
phase completes when its arrivals and its transaction bytes are both done, and a parity
wait passes as soon as the barrier's current phase has the other parity.

Copies land after random, heavy-tailed delays (so they complete out of issue order) and
consumers take random times.  The model checks that every consumer reads its own slab
fully landed and that no barrier receives more arrivals than its phase expects.  It finds
the fault when NS is not a multiple of wpg (a warp reaches round R of a stage whose round
R - 1 copy, another warp's, is still in flight, and the parity test passes) and none when
it is, the rule the kernel's host plan enforces."""
import heapq
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0          # index of the current (incomplete) phase
        self.over = False

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        if self.pending < 0:
            self.over = True
        self._maybe_complete()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe_complete()

    def parity_ready(self, parity):
        return (self.phase & 1) != parity


def simulate(NS, G, wpg, S, seed):
    """Returns the list of violations seen in one random schedule."""
    rng = random.Random(seed)
    full = [Bar(1) for _ in range(NS)]
    empty = [Bar(G) for _ in range(NS)]
    content = [None] * NS            # (slab, landed)
    bad = []
    events = []                      # (time, seq, kind, payload)
    seq = [0]

    def push(t, kind, payload):
        seq[0] += 1
        heapq.heappush(events, (t, seq[0], kind, payload))

    # actors poll when woken; a blocked actor is re-polled on every event
    prod = {"i": 0, "busy": 0.0}
    cons = {(g, w): {"i": w, "busy": 0.0, "reading": None} for g in range(G) for w in range(wpg)}
    t = 0.0
    for _ in range(200000):
        progressed = True
        while progressed:
            progressed = False
            # producer
            i = prod["i"]
            if i < S and prod["busy"] <= t:
                st, rd = i % NS, i // NS
                if rd == 0 or empty[st].parity_ready((rd - 1) & 1):
                    content[st] = (i, False)
                    full[st].arrive(tx=1)
                    delay = rng.uniform(1.0, 3.0) * (8.0 if rng.random() < 0.15 else 1.0)
                    push(t + delay, "land", (st, i))
                    prod["i"] += 1
                    prod["busy"] = t + 0.05
                    progressed = True
            # consumers
            for (g, w), c in cons.items():
                i = c["i"]
                if i >= S or c["busy"] > t or c["reading"] is not None:
                    continue
                st, rd = i % NS, i // NS
                if full[st].parity_ready(rd & 1):
                    if content[st] != (i, True):
                        bad.append(("read", g, w, i, content[st]))
                    c["reading"] = (st, i)
                    push(t + rng.uniform(0.3, 1.5), "done", (g, w))
                    progressed = True
        if not events:
            break
        t, _, kind, payload = heapq.heappop(events)
        if kind == "land":
            st, i = payload
            if content[st] == (i, False):
                content[st] = (i, True)
            else:
                bad.append(("overwritten", i, content[st]))
            full[st].complete_tx(1)
        else:
            g, w = payload
            c = cons[(g, w)]
            st, i = c["reading"]
            empty[st].arrive()
            c["reading"] = None
            c["i"] = i + wpg
    for b in full + empty:
        if b.over:
            bad.append(("over-arrival",))
    unfinished = prod["i"] < S or any(c["i"] < S for c in cons.values())
    if unfinished and not bad:
        bad.append(("stalled",))
    return bad


@pytest.mark.parametrize("NS,G,wpg", [(10, 4, 2), (20, 4, 2), (12, 4, 3), (4, 8, 2), (5, 8, 1),
                                      (24, 1, 8)])
def test_ring_is_exact_when_stages_are_a_multiple_of_wpg(NS, G, wpg):
    for seed in range(150):
        assert simulate(NS, G, wpg, S=6 * NS + 3, seed=seed) == [], (NS, G, wpg, seed)


@pytest.mark.parametrize("NS,G,wpg", [(11, 4, 2), (11, 4, 3), (5, 8, 2)])
def test_model_finds_the_parity_fault_otherwise(NS, G, wpg):
    """The stage counts of the three launch failures: the model must see the fault."""
    found = [simulate(NS, G, wpg, S=6 * NS + 3, seed=seed) for seed in range(150)]
    assert any(found)
