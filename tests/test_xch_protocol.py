"""A model of the post-norm GEMM's global row exchange, checked under random
interleavings and a weak memory (CPU only).

The kernel (the epilogue of nf_gemm_kernel with XCH_GLOBAL) runs a persistent
grid of G CTAs, all resident; tile t runs on CTA t mod G, in order.  Each CTA's
MMA fills one of two TMEM accumulators (tile j of a CTA uses buffer j mod 2 and
must wait until the epilogue has drained tile j - 2), and two epilogue groups
alternate tiles.  A tile's epilogue publishes its row partials as tagged words
(the launch's tag E + 1 beside each value), adds one to its row tile's counter,
polls that counter until all n_tiles column tiles of the row tile have counted,
then reads the row tile's partials, again while any word still carries an
older tag.  No fence orders the counter with the words: the model makes every
store visible after an arbitrary delay, each on its own, so a reader can see a
count before the words it stands for.

The scratch outlives launches: launch E counts in bank E & 1 and clears the
other bank (the previous launch's, whose row-tile count the header keeps);
every CTA counts itself in at the start and the last one advances E.

Checked: every tile reads exactly the partials of this launch's tiles of its
row tile, every schedule finishes, and a sequence of launches with changing
shapes reuses the scratch correctly.  Mutants that must be caught: a reader
that ignores the tags, a tag without the epoch, an epoch that never advances,
a launch that clears its own bank, and a grid below n_tiles / 2 CTAs.
"""
import random

import pytest

class Memory:
    """L2 as the threads see it: a store becomes visible after an arbitrary
    delay, independently of the others (a relaxed store, no fence)."""

    def __init__(self):
        self.vis = {}
        self.pending = []

    def store(self, addr, value):
        self.pending.append((addr, value))

    def add(self, addr, v):
        # a relaxed reduction: applied at L2 when it lands, in some order
        self.pending.append((addr, ("add", v)))

    def load(self, addr, default=0):
        return self.vis.get(addr, default)

    def land_one(self, rng):
        i = rng.randrange(len(self.pending))
        addr, value = self.pending.pop(i)
        if isinstance(value, tuple) and value[0] == "add":
            self.vis[addr] = self.vis.get(addr, 0) + value[1]
        else:
            self.vis[addr] = value

    def flush(self):
        # kernel boundary: everything the launch wrote is visible to the next
        while self.pending:
            self.land_one(random.Random(0))


class Deadlock(Exception):
    pass


def launch(mem, rng, m_tiles, n_tiles, grid, values, mutant=None, max_steps=200000):
    """One launch; returns {tile: partials read}.  values[(m, n)] is what tile
    (m, n) publishes in this launch."""
    E = mem.load(("hdr", 2))
    prev_rows = mem.load(("hdr", 3))
    tag = 0 if mutant == "tag_no_epoch" else E + 1
    bank = E & 1
    clear = bank if mutant == "clear_own_bank" else (E + 1) & 1
    tiles = m_tiles * n_tiles
    # start: every CTA clears its share of the other bank (relaxed stores that
    # may land at any time during the launch), then counts itself in; the
    # last one advances E (seen by the next launch, after this one ends)
    for c in range(grid):
        for i in range(c, prev_rows * 4, grid):
            mem.store(("cnt", clear, i), 0)
    if mutant != "epoch_stuck":
        mem.store(("hdr", 2), E + 1)
    mem.store(("hdr", 3), m_tiles)

    # per CTA: its tiles in order; per tile a state machine
    ctas = [[t for t in range(c, tiles, grid)] for c in range(grid)]
    drained = [[False] * len(seq) for seq in ctas]
    mma_done = [[False] * len(seq) for seq in ctas]
    # epilogue agent state per (cta, group): index into that group's tiles, phase
    epi = {(c, g): {"j": g, "phase": "wait_acc", "got": None} for c in range(grid) for g in (0, 1)}
    mma_next = [0] * grid
    result = {}

    def mma_step(c):
        j = mma_next[c]
        if j >= len(ctas[c]):
            return False
        if j >= 2 and not drained[c][j - 2]:
            return False  # accumulator j mod 2 still held by tile j - 2's epilogue
        mma_done[c][j] = True
        mma_next[c] += 1
        return True

    def epi_step(c, g):
        st = epi[(c, g)]
        j = st["j"]
        if j >= len(ctas[c]):
            return False
        t = ctas[c][j]
        m, n = divmod(t, n_tiles)
        if st["phase"] == "wait_acc":
            if not mma_done[c][j]:
                return False
            pa = values[(m, n)]
            mem.store(("part", m, n), (tag, pa))
            mem.add(("cnt", bank, m * 4), 1)
            st["phase"] = "wait_count"
            return True
        if st["phase"] == "wait_count":
            if mem.load(("cnt", bank, m * 4)) < n_tiles:
                return False
            st["phase"] = "gather"
            st["got"] = {}
            return True
        if st["phase"] == "gather":
            progressed = False
            for p in range(n_tiles):
                if p in st["got"]:
                    continue
                w = mem.load(("part", m, p), None)
                if w is None:
                    continue
                wtag, val = w
                if mutant == "ignore_tags" or wtag == tag:
                    st["got"][p] = val
                    progressed = True
            if len(st["got"]) < n_tiles:
                return progressed
            result[t] = [st["got"][p] for p in range(n_tiles)]
            drained[c][j] = True
            st["j"] = j + 2
            st["phase"] = "wait_acc"
            return True
        raise AssertionError(st)

    agents = [("mma", c) for c in range(grid)] + [("epi", c, g) for c in range(grid) for g in (0, 1)]
    for _ in range(max_steps):
        if all(st["j"] >= len(ctas[c]) for (c, g), st in epi.items()):
            break
        order = agents[:]
        rng.shuffle(order)
        moved = False
        # a random agent that can move moves; or a random store lands
        if mem.pending and rng.random() < 0.5:
            mem.land_one(rng)
            continue
        for a in order:
            if a[0] == "mma":
                moved = mma_step(a[1])
            else:
                moved = epi_step(a[1], a[2])
            if moved:
                break
        if not moved:
            if not mem.pending:
                raise Deadlock(f"no agent can move (grid {grid}, {m_tiles} x {n_tiles} tiles)")
            mem.land_one(rng)
    else:
        raise Deadlock("step limit")
    mem.flush()
    return result


def check(result, m_tiles, n_tiles, values):
    for t in range(m_tiles * n_tiles):
        m = t // n_tiles
        assert result[t] == [values[(m, p)] for p in range(n_tiles)], f"tile {t} read stale partials"


SHAPES = [(5, 3, 4), (8, 8, 4), (3, 16, 8), (12, 4, 7), (2, 2, 1), (9, 16, 16), (6, 5, 3)]


def run_sequence(seed, mutant=None, shapes=SHAPES, launches=3):
    rng = random.Random(seed)
    mem = Memory()
    for k in range(launches):
        for i, (m_tiles, n_tiles, grid) in enumerate(shapes):
            values = {(m, n): (seed, k, i, m, n) for m in range(m_tiles) for n in range(n_tiles)}
            result = launch(mem, rng, m_tiles, n_tiles, grid, values, mutant)
            check(result, m_tiles, n_tiles, values)


@pytest.mark.parametrize("seed", range(12))
def test_exchange_reads_this_launch_partials(seed):
    run_sequence(seed)


@pytest.mark.parametrize("mutant", ["ignore_tags", "tag_no_epoch", "epoch_stuck"])
def test_stale_partials_are_caught(mutant):
    # some schedule lets a reader see a count before the words it stands for
    with pytest.raises(AssertionError, match="stale"):
        for seed in range(40):
            run_sequence(seed, mutant)


def test_clearing_the_own_bank_is_caught():
    # the launch's counts are wiped while it counts: its waits never finish
    # (or a later launch passes them early, which the tags then absorb)
    with pytest.raises((Deadlock, AssertionError)):
        for seed in range(40):
            run_sequence(seed, "clear_own_bank")


def test_grid_rule():
    """2 G >= n_tiles never deadlocks; fewer CTAs can."""
    for seed in range(20):
        rng = random.Random(seed)
        for n_tiles in (2, 3, 5, 8, 16):
            grid = (n_tiles + 1) // 2
            values = {(m, n): (m, n) for m in range(4) for n in range(n_tiles)}
            check(launch(Memory(), rng, 4, n_tiles, grid, values), 4, n_tiles, values)
    with pytest.raises(Deadlock):
        # n_tiles 8 on 3 CTAs: a CTA's two accumulators both hold tiles of a
        # row tile whose other tiles wait behind them
        launch(Memory(), random.Random(1), 4, 8, 3, {(m, n): 0 for m in range(4) for n in range(8)})
