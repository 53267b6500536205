"""Host-side model of the forward kernels' two-thread MMA issue.

Where P has TMEM columns of its own (the one-tile kernel at D <= 128, the
two-tile kernel at D = 64), two threads issue the tensor-core products: one
the score products S = Q K^T, the other the products O += P V.  Products of
one thread complete in issue order, and a commit arrives once every earlier
product of the same thread is done; nothing orders one thread's products
against the other's.  So every reuse of a TMEM tile or a shared-memory slot
that one thread's product frees and the other thread's product (or the
softmax) refills needs a barrier of its own:

* one-tile: S_t goes into score tile t % 2 once the softmax warps hold
  S_{t-2} in registers (s_read), and the softmax stores P_j into P tile j % 2
  only after O += P_{j-2} V_{j-2} is done (pv_done); K slots are freed by the
  S thread, V slots by the PV thread;
* two-tile (D = 64): tile i's S_i(j+1) goes into its single score tile once
  the softmax of tile i holds S_i(j) in registers, P_i(j) is stored once
  O_i += P_i(j-1) V_{j-1} is done, and each K/V pair is released by a commit
  from each thread (a barrier expecting two arrivals);
* split rows (one tile, each row's keys split between two softmax halves):
  S_t goes into the single score tile once both halves hold S_{t-1} in
  registers (s_read expects both), and half h stores P_h(j) into its P tile
  j % 2 once O_h += P_h(j-2) V_{j-2} is done (tested early, waited for only
  when it was not yet done).

The model replays the producer, both MMA threads and the softmax warps with
copies landing in any order and the two threads' products completing in an
arbitrary interleaving, under mbarrier semantics (a parity wait succeeds for
any phase but the current one; a phase never takes more arrivals than it
expects), and checks that no tile or slot is rewritten while a product or the
softmax still needs it, that O is rescaled only after the last product into
it is done, and that the pipeline never deadlocks.  Tests keep five
plausible mistakes pinned as failing: the one-tile softmax storing P without
its pv_done wait (the single-thread kernel could rely on S_j's commit
instead), the two-tile S thread not waiting for s_read, a two-tile pair
release that expects one arrival instead of two, a split-row s_read that
expects one half only, and a split-row P store without its pv_done wait.
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


class _Machine:
    """Copies in flight, per-thread product queues, and the roles."""

    def __init__(self, seed):
        self.rnd = random.Random(seed)
        self.copies = []                 # (barrier, apply)
        self.queues = {"S": [], "PV": []}

    def step_async(self):
        """Complete one copy or the head of one thread's queue; False if none."""
        choices = []
        if self.copies:
            choices.append("copy")
        choices += [q for q, ops in self.queues.items() if ops]
        if not choices:
            return False
        pick = self.rnd.choice(choices)
        if pick == "copy":
            bar, apply = self.copies.pop(self.rnd.randrange(len(self.copies)))
            apply()
            bar.complete_tx(1)
        else:
            op = self.queues[pick].pop(0)   # one thread's products finish in issue order
            op()
        return True

    def run(self, roles, limit=400000):
        alive = [True] * len(roles)
        for _ in range(limit):
            busy = self.copies or any(self.queues.values())
            if not any(alive) and not busy:
                return
            if busy and (self.rnd.random() < 0.4 or not any(alive)):
                self.step_async()
                continue
            live = [i for i in range(len(roles)) if alive[i]]
            i = self.rnd.choice(live)
            try:
                next(roles[i])
            except StopIteration:
                alive[i] = False
        raise AssertionError("no progress: the pipeline deadlocked")


# ---------------------------------------------------------------- one-tile
def _run_onetile(n_kv, R, seed, skip_pv_wait=False):
    m = _Machine(seed)
    rnd = m.rnd
    k_full = [_Barrier() for _ in range(R)]
    k_empty = [_Barrier() for _ in range(R)]
    v_full = [_Barrier() for _ in range(R)]
    v_empty = [_Barrier() for _ in range(R)]
    s_full = [_Barrier(), _Barrier()]
    s_read = [_Barrier(), _Barrier()]
    p_full = [_Barrier(), _Barrier()]
    pv_done = [_Barrier(), _Barrier()]
    st = {"k_landed": {}, "v_landed": {}, "k_busy": {}, "v_busy": {},
          "s_tile": [None, None],      # score tile -> S index completed there
          "s_needed": [None, None],    # score tile -> S index the softmax has not read yet
          "p_tile": [None, None],      # P tile -> block stored
          "p_reader": [None, None],    # P tile -> block of the unfinished PV reading it
          "pv_last": -1}

    def producer():
        issued = {"k": 0, "v": 0}

        def load(kind):
            t = issued[kind]
            full, empty = (k_full, k_empty) if kind == "k" else (v_full, v_empty)
            busy, landed = (st["k_busy"], st["k_landed"]) if kind == "k" else (st["v_busy"], st["v_landed"])
            if t >= R:
                while not empty[t % R].passed(((t - R) // R) & 1):
                    yield
            assert busy.get(t % R, 0) == 0, f"copy of {kind}{t} into a slot still read"
            landed.pop(t % R, None)
            full[t % R].arrive(tx=1)
            m.copies.append((full[t % R], lambda s=t % R, t=t, landed=landed: landed.__setitem__(s, t)))
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

    def s_thread():
        def next_s(t):
            while not k_full[t % R].passed((t // R) & 1):
                yield
            assert st["k_landed"].get(t % R) == t, f"S_{t} issued before K_{t} landed"
            assert st["s_needed"][t & 1] is None, f"S_{t} written over S_{t - 2} before the softmax read it"
            st["k_busy"][t % R] = st["k_busy"].get(t % R, 0) + 1

            def done(t=t):
                st["s_tile"][t & 1] = t
                st["s_needed"][t & 1] = t
            q = m.queues["S"]
            q.append(done)
            q.append(lambda t=t: s_full[t & 1].arrive())
            q.append(lambda s=t % R: (st["k_busy"].__setitem__(s, st["k_busy"][s] - 1), k_empty[s].arrive()))

        yield from next_s(0)
        if n_kv > 1:
            yield from next_s(1)
        for t in range(2, n_kv):
            while not s_read[t & 1].passed(((t - 2) >> 1) & 1):
                yield
            yield from next_s(t)
            yield

    def pv_thread():
        for j in range(n_kv):
            while not (v_full[j % R].passed((j // R) & 1) and p_full[j & 1].passed((j >> 1) & 1)):
                yield
            assert st["v_landed"].get(j % R) == j, f"PV_{j} issued before V_{j} landed"
            assert st["p_tile"][j & 1] == j, f"PV_{j} reads P tile without P_{j}"
            st["v_busy"][j % R] = st["v_busy"].get(j % R, 0) + 1
            st["p_reader"][j & 1] = j

            def done(j=j):
                st["pv_last"] = j
                st["p_reader"][j & 1] = None
            q = m.queues["PV"]
            q.append(done)
            q.append(lambda s=j % R: (st["v_busy"].__setitem__(s, st["v_busy"][s] - 1), v_empty[s].arrive()))
            q.append(lambda j=j: pv_done[j & 1].arrive())
            yield

    def softmax():
        for j in range(n_kv):
            while not s_full[j & 1].passed((j >> 1) & 1):
                yield
            assert st["s_tile"][j & 1] == j, f"softmax of block {j} read a score tile without S_{j}"
            st["s_needed"][j & 1] = None          # S_j is in registers now
            s_read[j & 1].arrive()
            yield
            if rnd.random() < 0.3 and j > 0:      # the lazy max moves: O is rescaled
                while not pv_done[(j - 1) & 1].passed(((j - 1) >> 1) & 1):
                    yield
                assert st["pv_last"] >= j - 1, "O rescaled while O += P V still runs"
            if j >= 2 and not skip_pv_wait:
                while not pv_done[j & 1].passed(((j - 2) >> 1) & 1):
                    yield
            assert st["p_reader"][j & 1] is None, f"P_{j} written while a product still reads tile {j & 1}"
            st["p_tile"][j & 1] = j
            p_full[j & 1].arrive()
            yield

    m.run([producer(), s_thread(), pv_thread(), softmax()])


@pytest.mark.parametrize("R", [3, 4])
@pytest.mark.parametrize("n_kv", [1, 2, 3, 4, 5, 8, 13])
def test_onetile_two_threads_hold_their_invariants(R, n_kv):
    for seed in range(40):
        _run_onetile(n_kv, R, seed)


def _caught(run, cases, seeds=200):
    """True once some seeded run of a planted mistake trips an invariant."""
    for case in cases:
        for seed in range(seeds):
            try:
                run(case, seed)
            except AssertionError:
                return True
    return False


def test_onetile_p_store_without_its_pv_wait_is_caught():
    assert _caught(lambda n, seed: _run_onetile(n, 3, seed, skip_pv_wait=True), (4, 6, 9))


# ---------------------------------------------------------------- two-tile, D = 64
def _run_twotile(n_kv, slots, seed, skip_s_read=False, release_count=2):
    m = _Machine(seed)
    rnd = m.rnd
    pairs = slots // 2
    full = [_Barrier() for _ in range(pairs)]
    empty = [_Barrier(release_count) for _ in range(pairs)]
    s_full = [_Barrier(), _Barrier()]
    s_read = [_Barrier(), _Barrier()]
    p_full = [_Barrier(), _Barrier()]
    pv_done = [_Barrier(), _Barrier()]
    st = {"landed": {}, "busy": {},
          "s_tile": [None, None], "s_needed": [None, None],
          "p_tile": [None, None], "p_reader": [None, None],
          "pv_last": [-1, -1]}

    def tiles_of(mm):
        out = []
        if mm >= 1:
            out.append(((2 * mm - 1) % slots, ("V", mm - 1)))
        if mm < n_kv:
            out.append(((2 * mm) % slots, ("K", mm)))
        return out

    def producer():
        armed = 0
        for mm in range(n_kv + 1):
            if mm >= pairs:
                pm = mm - pairs
                while not empty[pm % pairs].passed((pm // pairs) & 1):
                    yield
            tiles = tiles_of(mm)
            bar = full[mm % pairs]
            bar.arrive(tx=len(tiles))
            for slot, tile in tiles:
                assert st["busy"].get(slot, 0) == 0, f"copy of {tile} into slot {slot} while it is still read"
                st["landed"].pop(slot, None)
                m.copies.append((bar, lambda s=slot, t=tile: st["landed"].__setitem__(s, t)))
            armed = mm + 1
            yield
        for mm in range(max(0, armed - pairs), armed):
            while not full[mm % pairs].passed((mm // pairs) & 1):
                yield

    def use(slot):
        st["busy"][slot] = st["busy"].get(slot, 0) + 1

    def free(slot):
        st["busy"][slot] -= 1

    def s_thread():
        q = m.queues["S"]

        def issue_s(i, j, slot):
            assert st["landed"].get(slot) == ("K", j), f"S_{i}({j}) issued before K_{j} landed"
            assert st["s_needed"][i] is None, f"S_{i}({j}) written over S_{i}({j - 1}) before the softmax read it"
            use(slot)

            def done(i=i, j=j, slot=slot):
                st["s_tile"][i] = j
                st["s_needed"][i] = j
                free(slot)
            q.append(done)
            q.append(lambda i=i: s_full[i].arrive())

        while not full[0].passed(0):
            yield
        issue_s(0, 0, 0)
        issue_s(1, 0, 0)
        q.append(lambda: empty[0].arrive())
        for j in range(n_kv):
            if j + 1 < n_kv:
                mm = j + 1
                while not full[mm % pairs].passed((mm // pairs) & 1):
                    yield
                for i in range(2):
                    if not skip_s_read:
                        while not s_read[i].passed(j & 1):
                            yield
                    issue_s(i, j + 1, (2 * j + 2) % slots)
            q.append(lambda mm=j + 1: empty[mm % pairs].arrive())
            yield

    def pv_thread():
        q = m.queues["PV"]
        q.append(lambda: empty[0].arrive())
        for j in range(n_kv):
            mm = j + 1
            while not full[mm % pairs].passed((mm // pairs) & 1):
                yield
            slot = (2 * j + 1) % slots
            for i in range(2):
                while not p_full[i].passed(j & 1):
                    yield
                assert st["landed"].get(slot) == ("V", j), f"PV_{i}({j}) issued before V_{j} landed"
                assert st["p_tile"][i] == j, f"PV_{i}({j}) reads P_{i} without block {j}"
                use(slot)
                st["p_reader"][i] = j

                def done(i=i, j=j, slot=slot):
                    st["pv_last"][i] = j
                    st["p_reader"][i] = None
                    free(slot)
                q.append(done)
                q.append(lambda i=i: pv_done[i].arrive())
            q.append(lambda mm=mm: empty[mm % pairs].arrive())
            yield

    def softmax(i):
        for j in range(n_kv):
            while not s_full[i].passed(j & 1):
                yield
            assert st["s_tile"][i] == j, f"softmax {i} of block {j} read a score tile without S_{i}({j})"
            st["s_needed"][i] = None
            s_read[i].arrive()
            yield
            if j > 0:
                # before the first P store (and any O rescale) PV_i(j-1) is done
                while not pv_done[i].passed((j - 1) & 1):
                    yield
                if rnd.random() < 0.3:
                    assert st["pv_last"][i] >= j - 1, "O rescaled while O += P V still runs"
            assert st["p_reader"][i] is None, f"P_{i}({j}) written while a product still reads it"
            st["p_tile"][i] = j
            p_full[i].arrive()
            yield

    m.run([producer(), s_thread(), pv_thread(), softmax(0), softmax(1)])


@pytest.mark.parametrize("n_kv", [1, 2, 3, 4, 5, 7, 9, 16])
def test_twotile_two_threads_hold_their_invariants(n_kv):
    for seed in range(50):
        _run_twotile(n_kv, 8, seed)


def test_twotile_s_issue_without_s_read_is_caught():
    assert _caught(lambda n, seed: _run_twotile(n, 8, seed, skip_s_read=True), (3, 5, 8))


def test_twotile_pair_release_expecting_one_arrival_is_caught():
    assert _caught(lambda n, seed: _run_twotile(n, 8, seed, release_count=1), (6, 9, 16))


# ---------------------------------------------------------------- split rows
def _run_halves(n_kv, R, seed, s_read_count=2, skip_p_wait=False):
    """The split-row kernel: one score tile S read by both key halves' softmax
    warps (s_read expects both), P tiles per half and parity of the block,
    pv_done per half and P tile, K freed by the S thread and V by the PV
    thread.  The softmax tests pv_done early and waits only if needed."""
    m = _Machine(seed)
    rnd = m.rnd
    k_full = [_Barrier() for _ in range(R)]
    k_empty = [_Barrier() for _ in range(R)]
    v_full = [_Barrier() for _ in range(R)]
    v_empty = [_Barrier() for _ in range(R)]
    s_full = _Barrier()
    s_read = _Barrier(s_read_count)
    p_full = [[_Barrier(), _Barrier()], [_Barrier(), _Barrier()]]      # [half][P tile]
    pv_done = [[_Barrier(), _Barrier()], [_Barrier(), _Barrier()]]
    st = {"k_landed": {}, "v_landed": {}, "k_busy": {}, "v_busy": {},
          "s_tile": None, "s_unread": set(),
          "p_tile": [[None, None], [None, None]], "p_reader": [[None, None], [None, None]],
          "pv_last": [-1, -1]}

    def producer():
        issued = {"k": 0, "v": 0}

        def load(kind):
            t = issued[kind]
            full, empty = (k_full, k_empty) if kind == "k" else (v_full, v_empty)
            busy, landed = (st["k_busy"], st["k_landed"]) if kind == "k" else (st["v_busy"], st["v_landed"])
            if t >= R:
                while not empty[t % R].passed(((t - R) // R) & 1):
                    yield
            assert busy.get(t % R, 0) == 0, f"copy of {kind}{t} into a slot still read"
            landed.pop(t % R, None)
            full[t % R].arrive(tx=1)
            m.copies.append((full[t % R], lambda s=t % R, t=t, landed=landed: landed.__setitem__(s, t)))
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

    def s_thread():
        for t in range(n_kv):
            while not k_full[t % R].passed((t // R) & 1):
                yield
            if t > 0:
                while not s_read.passed((t - 1) & 1):
                    yield
            assert st["k_landed"].get(t % R) == t, f"S_{t} issued before K_{t} landed"
            assert not st["s_unread"], f"S_{t} written before both halves read S_{t - 1}"
            st["k_busy"][t % R] = st["k_busy"].get(t % R, 0) + 1

            def done(t=t):
                st["s_tile"] = t
                st["s_unread"] = {0, 1}
            q = m.queues["S"]
            q.append(done)
            q.append(lambda: s_full.arrive())
            q.append(lambda s=t % R: (st["k_busy"].__setitem__(s, st["k_busy"][s] - 1), k_empty[s].arrive()))
            yield

    def pv_thread():
        q = m.queues["PV"]
        for j in range(n_kv):
            buf = j & 1
            while not v_full[j % R].passed((j // R) & 1):
                yield
            for h in range(2):
                while not p_full[h][buf].passed((j >> 1) & 1):
                    yield
                assert st["v_landed"].get(j % R) == j, f"PV_{h}({j}) issued before V_{j} landed"
                assert st["p_tile"][h][buf] == j, f"PV_{h}({j}) reads a P tile without P_{h}({j})"
                st["v_busy"][j % R] = st["v_busy"].get(j % R, 0) + 1
                st["p_reader"][h][buf] = j

                def done(h=h, j=j, buf=buf):
                    st["pv_last"][h] = j
                    st["p_reader"][h][buf] = None
                    st["v_busy"][j % R] -= 1
                q.append(done)
                q.append(lambda h=h, buf=buf: pv_done[h][buf].arrive())
            q.append(lambda s=j % R: v_empty[s].arrive())
            yield

    def softmax(h):
        for j in range(n_kv):
            buf = j & 1
            while not s_full.passed(j & 1):
                yield
            assert st["s_tile"] == j and h in st["s_unread"], f"half {h} of block {j} read a score tile without S_{j}"
            p_free = j < 2 or pv_done[h][buf].passed(((j - 2) >> 1) & 1)
            st["s_unread"].discard(h)
            s_read.arrive()
            yield
            if j > 0 and rnd.random() < 0.3:       # the lazy max moves: O_h is rescaled
                while not pv_done[h][(j - 1) & 1].passed(((j - 1) >> 1) & 1):
                    yield
                assert st["pv_last"][h] >= j - 1, "O_h rescaled while O_h += P V still runs"
            if not p_free and not skip_p_wait:
                while not pv_done[h][buf].passed(((j - 2) >> 1) & 1):
                    yield
            assert st["p_reader"][h][buf] is None, f"P_{h}({j}) written while a product still reads its tile"
            st["p_tile"][h][buf] = j
            p_full[h][buf].arrive()
            yield

    m.run([producer(), s_thread(), pv_thread(), softmax(0), softmax(1)])


@pytest.mark.parametrize("R", [3, 4])
@pytest.mark.parametrize("n_kv", [1, 2, 3, 4, 5, 8, 13])
def test_split_rows_hold_their_invariants(R, n_kv):
    for seed in range(40):
        _run_halves(n_kv, R, seed)


def test_split_rows_s_read_from_one_half_is_caught():
    assert _caught(lambda n, seed: _run_halves(n, 3, seed, s_read_count=1), (3, 5, 8))


def test_split_rows_p_store_without_its_pv_wait_is_caught():
    assert _caught(lambda n, seed: _run_halves(n, 3, seed, skip_p_wait=True), (4, 6, 9))
