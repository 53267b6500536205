"""Host-side model of the forward kernel's K/V ring synchronisation.

The two-tile forward kernel streams K_j and V_j through a ring of S
shared-memory slots (K_j in slot 2j mod S, V_j in slot 2j+1 mod S; S = 4 at
D = 128, 8 at D = 64).  Its MMA warp reads V_j (for P V_j) and K_{j+1} (for
the next score tile) in the same iteration, so the tiles move in pairs:
pair m = (V_{m-1}, K_m), with K_0 alone as pair 0 and the last V alone as the
last pair.  Each pair has a "full" barrier (one arrival with the bytes of its
copies) and an "empty" barrier (one commit from the MMA warp once both of its
tiles are read).  Pair m fills the slots of pair m - S/2, so the producer
waits for that pair's release first; both kinds of barrier are used
round-robin over S/2.

This model replays the producer warp, the MMA warp and the asynchronous
completions (TMA copies landing, MMA commits completing) in random orders,
with mbarrier semantics (one expected arrival per phase, a transaction count,
and a parity wait that succeeds for any phase other than the current one), and
checks what the kernel relies on:

* no phase of a barrier receives a second arrival;
* no copy goes into a slot whose previous tile the MMA warp still reads;
* every MMA-side wait returns only after the tiles it covers have landed;
* the producer's final drain returns only after every copy has landed;
* the pipeline always finishes (no deadlock).

A test also keeps a plausible mistake pinned as failing: waiting for the
release of a pair one older than the one whose slots pair m fills.
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

    def arrive_expect_tx(self, n):
        if self.pending <= 0:
            raise AssertionError("second arrival in one phase")
        self.tx += n
        self.pending -= 1
        self._advance()

    def arrive(self):
        if self.pending <= 0:
            raise AssertionError("second arrival in one phase")
        self.pending -= 1
        self._advance()

    def complete_tx(self, n):
        self.tx -= n
        self._advance()

    def passed(self, parity):
        return (self.phase & 1) != parity


def _run(n_kv, slots, seed, release_lag=None):
    """One randomised run; release_lag: which earlier pair's release the
    producer waits for before filling pair m (the kernel: slots // 2)."""
    pairs = slots // 2
    lag = pairs if release_lag is None else release_lag
    rnd = random.Random(seed)
    full = [_Barrier() for _ in range(pairs)]
    empty = [_Barrier() for _ in range(pairs)]
    landed = {}          # slot -> tile that has fully landed there
    busy = set()         # slots whose tile the MMA warp may still read
    copies = []          # TMA copies in flight
    commits = []         # MMA commits not yet completed: the slots they release

    def tiles_of(m):
        out = []
        if m >= 1:
            out.append(((2 * m - 1) % slots, ("V", m - 1)))
        if m < n_kv:
            out.append(((2 * m) % slots, ("K", m)))
        return out

    def producer():
        armed = 0
        for m in range(n_kv + 1):
            if m >= lag:
                pm = m - lag
                while not empty[pm % pairs].passed((pm // pairs) & 1):
                    yield
            tiles = tiles_of(m)
            bar = full[m % pairs]
            bar.arrive_expect_tx(len(tiles))
            for slot, tile in tiles:
                assert slot not in busy, f"copy of {tile} into slot {slot} while it is still read"
                busy.add(slot)
                landed.pop(slot, None)
                copies.append((bar, slot, tile))
            armed = m + 1
            yield
        for m in range(max(0, armed - pairs), armed):
            while not full[m % pairs].passed((m // pairs) & 1):
                yield
        assert not copies, "drain passed with copies in flight"

    def mma():
        while not full[0].passed(0):
            yield
        assert landed.get(0) == ("K", 0)
        commits.append((0, [0]))
        for j in range(n_kv):
            m = j + 1
            while not full[m % pairs].passed((m // pairs) & 1):
                yield
            for slot, tile in tiles_of(m):
                assert landed.get(slot) == tile, f"{tile} read before it landed"
            commits.append((m % pairs, [slot for slot, _ in tiles_of(m)]))
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
                idx, freed = commits.pop(0)      # commits complete in issue order
                busy.difference_update(freed)
                empty[idx].arrive()
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
        _run(n_kv, slots, seed)


def test_waiting_for_the_wrong_release_breaks_the_ring():
    failures = 0
    for n_kv in (3, 5, 8):
        for seed in range(200):
            try:
                _run(n_kv, 4, seed, release_lag=3)
            except AssertionError:
                failures += 1
    assert failures > 0
