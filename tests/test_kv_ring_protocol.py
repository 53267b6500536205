"""Host-side model of the forward kernel's K/V ring synchronisation.

The two-tile forward kernel streams K_j and V_j through a ring of shared-memory
slots (K_j in slot 2j mod S, V_j in slot 2j+1 mod S, S = 4 at D = 128, 8 at
D = 64).  Its MMA warp reads V_j (for P V_j) and then K_{j+1} (for the next
score tile) back to back, so one arrival barrier covers the pair
(V_j, K_{j+1}) -- "pair j+1" -- and K_0 alone is pair 0.  The barriers are used
round-robin; the kernel keeps S/2 + 1 of them.

This model replays the producer warp, the MMA warp and the asynchronous
completions (TMA copies landing, MMA commits freeing slots) in random orders,
with mbarrier semantics (one expected arrival per phase, a transaction count,
and a parity wait that succeeds for any phase other than the current one), and
checks what the kernel relies on:

* no phase of a barrier receives a second arrival;
* every MMA-side wait returns only after the tiles it covers have landed;
* the producer's final drain returns only after every copy has landed;
* the pipeline always finishes (no deadlock).

With only S/2 barriers, pair S/2 is armed by a V tile that goes into a fresh
slot, so nothing makes it wait for pair 0 to complete on the same barrier: the
model shows the resulting double arrival, and a test keeps that reading pinned.
"""
import random

import pytest


class _Barrier:
    def __init__(self):
        self.phase = 0
        self.pending = 1
        self.tx = 0

    def _advance(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = 1

    def arrive(self):
        if self.pending <= 0:
            raise AssertionError("second arrival in one phase")
        self.pending -= 1
        self._advance()

    def expect_tx(self, n):
        self.tx += n

    def complete_tx(self, n):
        self.tx -= n
        self._advance()

    def passed(self, parity):
        return (self.phase & 1) != parity


def _run(n_kv, slots, pair_bars, seed):
    rnd = random.Random(seed)
    pair = [_Barrier() for _ in range(pair_bars)]
    empty = [_Barrier() for _ in range(slots)]
    landed = {}          # slot -> tile that has fully landed there
    copies = []          # TMA copies in flight
    commits = []         # MMA commits not yet completed

    def producer():
        armed = 0
        for j in range(n_kv):
            for w in range(2):
                idx = 2 * j + w
                slot, rnd_ = idx % slots, idx // slots
                if rnd_ > 0:
                    while not empty[slot].passed((rnd_ - 1) & 1):
                        yield
                m = j + w
                bar = pair[m % pair_bars]
                closes = w == 0 or j + 1 == n_kv
                bar.expect_tx(1)
                if closes:
                    bar.arrive()
                landed.pop(slot, None)
                copies.append((bar, slot, ("KV"[w], j)))
                armed = m + 1
                yield
        for m in range(max(0, armed - pair_bars), armed):
            while not pair[m % pair_bars].passed((m // pair_bars) & 1):
                yield
        assert not copies, "drain passed with copies in flight"

    def mma():
        while not pair[0].passed(0):
            yield
        assert landed.get(0) == ("K", 0)
        commits.append(0)
        for j in range(n_kv):
            slot_v, slot_k = (2 * j + 1) % slots, (2 * j + 2) % slots
            more = j + 1 < n_kv
            m = j + 1
            while not pair[m % pair_bars].passed((m // pair_bars) & 1):
                yield
            assert landed.get(slot_v) == ("V", j), f"P V_{j} issued before V_{j} landed"
            if more:
                assert landed.get(slot_k) == ("K", j + 1), f"S_{j + 1} issued before K_{j + 1} landed"
            commits.append(slot_v)
            if more:
                commits.append(slot_k)
            yield

    roles = [producer(), mma()]
    alive = [True, True]
    for _ in range(100000):
        if not any(alive) and not copies and not commits:
            return
        if (copies or commits) and (rnd.random() < 0.4 or not any(alive)):
            if copies and (not commits or rnd.random() < 0.5):
                bar, slot, tile = copies.pop(rnd.randrange(len(copies)))
                landed[slot] = tile
                bar.complete_tx(1)
            else:
                empty[commits.pop(rnd.randrange(len(commits)))].arrive()
            continue
        live = [i for i in range(2) if alive[i]]
        if not live:
            continue
        i = rnd.choice(live)
        try:
            next(roles[i])
        except StopIteration:
            alive[i] = False
    raise AssertionError("no progress: the pipeline deadlocked")


@pytest.mark.parametrize("slots", [4, 8])
@pytest.mark.parametrize("n_kv", [1, 2, 3, 4, 5, 7, 9, 16])
def test_pair_barriers_hold_their_invariants(slots, n_kv):
    for seed in range(150):
        _run(n_kv, slots, slots // 2 + 1, seed)


def test_one_barrier_fewer_breaks_the_ring():
    failures = 0
    for n_kv in (2, 4, 6):
        for seed in range(200):
            try:
                _run(n_kv, 4, 2, seed)
            except AssertionError:
                failures += 1
    assert failures > 0
