"""Host-side model of the one-tile forward kernel's synchronisation.

The one-tile kernel (one 128-row query tile per CTA) streams K_t and V_t
through two rings of R shared-memory slots each (K_t in K slot t % R, V_t in
V slot t % R), keeps two score tiles S_0, S_1 and two P tiles in tensor
memory, and issues its MMAs from one thread in the order S_0, S_1, then per
key block j: O += P_j V_j, followed by S_{j+2} into score tile j % 2.  (At
head dimension 256 P is written over its score tile and S_{j+1} is issued
before O += P_j V_j instead.)  Barriers: per slot a "full" (copy landed) and
an "empty" (MMA commit after the last product reading it) barrier, per score
tile s_full, per P tile p_full (the softmax hands P_j over) and pv_done (the
product reading P_j has completed).

The model replays the producer warp, the MMA warp and the softmax warps with
asynchronous completions (copies landing in any order, tensor-core ops
completing in issue order, a commit arriving once every earlier op is done)
under mbarrier semantics (one arrival per phase; a parity wait succeeds for
any phase other than the current one) and checks:

* no copy goes into a slot an issued, unfinished product still reads;
* every product reads operands that have landed: K_t, V_j, P_j, S_j;
* S_{t} is not written while the softmax still has to read S_{t-2};
* P_j is not written while the product reading P_{j-2} is unfinished;
* an O rescale at block j happens after O += P_{j-1} V_{j-1} is done;
* the pipeline finishes (no deadlock), and the producer's drain waits for
  every copy.

The softmax does not wait for O += P_{j-2} V_{j-2} before rewriting P tile
j % 2: S_j is issued after that product, and the commit that completes S_j
covers every earlier op of the issuing thread, so the s_full wait of block j
already implies it.  A test keeps the mistake that would break this pinned
as failing: issuing S_{j+2} before O += P_j V_j.
"""
import random

import pytest


class _Barrier:
    def __init__(self, count=1):
        self.count = count
        self.phase = 0
        self.pending = count
        self.tx = 0

    def _advance(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, tx=0):
        if self.pending <= 0:
            raise AssertionError("extra arrival in one phase")
        self.tx += tx
        self.pending -= 1
        self._advance()

    def complete_tx(self, n):
        self.tx -= n
        self._advance()

    def passed(self, parity):
        return (self.phase & 1) != parity


def _run(n_kv, R, p_apart, seed, s_before_pv=False):
    rnd = random.Random(seed)
    k_full = [_Barrier() for _ in range(R)]
    k_empty = [_Barrier() for _ in range(R)]
    v_full = [_Barrier() for _ in range(R)]
    v_empty = [_Barrier() for _ in range(R)]
    s_full = [_Barrier(), _Barrier()]
    p_full = [_Barrier(), _Barrier()]
    pv_done = [_Barrier(), _Barrier()]
    k_landed, v_landed = {}, {}          # slot -> tile index landed there
    k_busy, v_busy = {}, {}              # slot -> number of unfinished products reading it
    copies = []                          # (kind, slot, t)
    ops = []                             # tensor-core queue: ("S", t) / ("PV", j) / ("commit", bar)
    state = {"s_tile": [None, None],     # score tile -> S index written (completed)
             "s_read": -1,               # last block whose S the softmax has read
             "p_tile": [None, None],     # P tile -> block index stored
             "pv_done": -1,              # last completed O += P V
             "p_reader": [None, None]}   # P tile -> block of the unfinished product reading it

    def col_s(t):
        return t & 1

    def producer():
        issued = {"k": 0, "v": 0}

        def load(kind):
            t = issued[kind]
            full, empty = (k_full, k_empty) if kind == "k" else (v_full, v_empty)
            busy, landed = (k_busy, k_landed) if kind == "k" else (v_busy, v_landed)
            if t >= R:
                while not empty[t % R].passed(((t - R) // R) & 1):
                    yield
            assert busy.get(t % R, 0) == 0, f"copy of {kind}{t} into a slot still read"
            landed.pop(t % R, None)
            full[t % R].arrive(tx=1)
            copies.append((kind, t % R, t))
            issued[kind] += 1

        yield from load("k")
        if n_kv > 1:
            yield from load("k")
        while issued["v"] < n_kv:
            yield from load("v")
            if issued["k"] < n_kv:
                yield from load("k")
            yield
        for kind, full in (("k", k_full), ("v", v_full)):
            for t in range(max(0, issued[kind] - R), issued[kind]):
                while not full[t % R].passed((t // R) & 1):
                    yield
        assert not copies, "drain passed with copies in flight"

    def mma():
        def next_s(t):
            while not k_full[t % R].passed((t // R) & 1):
                yield
            assert k_landed.get(t % R) == t, f"S_{t} issued before K_{t} landed"
            # the score tile must have been read by the softmax (S_{t-2})
            assert state["s_read"] >= t - 2, f"S_{t} written over S_{t-2} before the softmax read it"
            k_busy[t % R] = k_busy.get(t % R, 0) + 1
            ops.append(("S", t))
            ops.append(("commit", s_full[col_s(t)]))
            ops.append(("commit_k", t % R))

        yield from next_s(0)
        if p_apart and n_kv > 1:
            yield from next_s(1)
        for j in range(n_kv):
            if not p_apart and j + 1 < n_kv:
                yield from next_s(j + 1)
            if p_apart and s_before_pv and j + 2 < n_kv:
                while not p_full[j & 1].passed((j >> 1) & 1):
                    yield
                yield from next_s(j + 2)
            while not (v_full[j % R].passed((j // R) & 1) and p_full[j & 1].passed((j >> 1) & 1)):
                yield
            assert v_landed.get(j % R) == j, f"PV_{j} issued before V_{j} landed"
            assert state["p_tile"][j & 1] == j, f"PV_{j} reads P tile without P_{j}"
            v_busy[j % R] = v_busy.get(j % R, 0) + 1
            state["p_reader"][j & 1] = j
            ops.append(("PV", j))
            ops.append(("commit_v", j % R))
            ops.append(("commit", pv_done[j & 1]))
            if p_apart and not s_before_pv and j + 2 < n_kv:
                yield from next_s(j + 2)
            yield

    def softmax():
        for j in range(n_kv):
            while not s_full[j & 1].passed((j >> 1) & 1):
                yield
            assert state["s_tile"][j & 1] == j, f"softmax of block {j} read a score tile without S_{j}"
            if rnd.random() < 0.3 and j > 0:          # the lazy max moves: O is rescaled
                while not pv_done[(j - 1) & 1].passed(((j - 1) >> 1) & 1):
                    yield
                assert state["pv_done"] >= j - 1, "O rescaled while O += P V still runs"
            tile = j & 1 if p_apart else col_s(j)
            assert state["p_reader"][tile] is None, f"P_{j} written while a product still reads tile {tile}"
            state["s_read"] = j
            state["p_tile"][tile] = j
            p_full[j & 1].arrive()
            yield

    roles = [producer(), mma(), softmax()]
    alive = [True, True, True]
    for _ in range(200000):
        if not any(alive) and not copies and not ops:
            return
        if (copies or ops) and (rnd.random() < 0.4 or not any(alive)):
            if copies and (not ops or rnd.random() < 0.5):
                kind, slot, t = copies.pop(rnd.randrange(len(copies)))
                (k_landed if kind == "k" else v_landed)[slot] = t
                (k_full if kind == "k" else v_full)[slot].complete_tx(1)
            else:
                op = ops.pop(0)                        # tensor-core ops finish in issue order
                if op[0] == "S":
                    state["s_tile"][col_s(op[1])] = op[1]
                elif op[0] == "PV":
                    state["pv_done"] = op[1]
                    state["p_reader"][op[1] & 1] = None
                elif op[0] == "commit_k":
                    k_busy[op[1]] -= 1
                    k_empty[op[1]].arrive()
                elif op[0] == "commit_v":
                    v_busy[op[1]] -= 1
                    v_empty[op[1]].arrive()
                else:
                    op[1].arrive()
            continue
        live = [i for i in range(3) if alive[i]]
        if not live:
            continue
        i = rnd.choice(live)
        try:
            next(roles[i])
        except StopIteration:
            alive[i] = False
    raise AssertionError("no progress: the pipeline deadlocked")


@pytest.mark.parametrize("R,p_apart", [(3, True), (4, True), (1, False)])
@pytest.mark.parametrize("n_kv", [1, 2, 3, 4, 5, 8, 13])
def test_onetile_barriers_hold_their_invariants(R, p_apart, n_kv):
    for seed in range(120):
        _run(n_kv, R, p_apart, seed)


def test_scores_issued_before_the_product_reading_p_break_the_p_tiles():
    failures = 0
    for n_kv in (4, 6, 9):
        for seed in range(200):
            try:
                _run(n_kv, 3, True, seed, s_before_pv=True)
            except AssertionError:
                failures += 1
    assert failures > 0
