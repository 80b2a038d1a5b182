"""A model of the FlashNormAttention forward kernel's synchronisation, checked
under random interleavings (CPU only).

The persistent kernel (one CTA of a cluster; the cluster's CTAs run the same
sequence, so the cross-CTA exchanges add no ordering the model needs) has a
TMA producer and NG compute groups, each with its MMA warp, that talk through
mbarriers waited on by phase PARITY.  A parity wait for completion #c is only
correct if, every time it is evaluated, the barrier has completed c or c + 1
phases: at c - 1 or fewer the parity reads an older phase as done, at c + 2 or
more it waits for a phase that may never come.  The model encodes the
protocol's waits and arrivals in the kernel's order and checks that rule for
every wait and try-wait, that every arrival counts toward the phase it is meant
for, that K and V are never replaced under a tile still to use them, and that
every schedule finishes.

A variant with the first persistent producer's rule (waiting, at a batch
switch, on each group's per-tile O barrier for its last tile) must be caught.
"""
import random

import pytest

NQ = 4          # q tile buffers
END = None      # end record


class Bar:
    """An mbarrier: completed phases and arrivals in the current phase."""

    def __init__(self, name, count=1):
        self.name, self.count, self.done, self.arrivals = name, count, 0, 0

    def arrive(self, phase):
        assert self.done == phase, f"{self.name}: arrival for phase {phase} while at phase {self.done}"
        self.arrivals += 1
        if self.arrivals == self.count:
            self.done += 1
            self.arrivals = 0


class Violation(Exception):
    pass


class State:
    def __init__(self, ng):
        self.ng = ng
        self.qfull = [Bar(f"qfull{j}") for j in range(NQ)]
        self.qempty = [Bar(f"qempty{j}") for j in range(NQ)]
        self.kvload = Bar("kv")
        self.kvfree = Bar("kvfree", count=ng)
        self.ofull = [Bar(f"ofull{g}") for g in range(ng)]
        self.rec = [None] * NQ
        self.kv_in_buffer = -1          # the last K/V load issued into the single buffer
        self.inflight = {}              # group -> kv of the tile whose MMAs are in flight


def check_parity(bar, c):
    """The rule for a parity wait on completion #c, at evaluation time."""
    if not (c <= bar.done <= c + 1):
        raise Violation(f"{bar.name}: parity wait for completion {c} evaluated at {bar.done} completed")


def producer(st, batches, rule="current"):
    ng, t, kv_loads = st.ng, 0, 0
    for T in batches:
        if T == 0:
            continue
        kv, t_first, m = kv_loads, t, 0
        # tiles whose buffer is already free go first (non-blocking try-waits),
        # once the previous K/V load has landed
        while m < T and t < t_first + NQ and rule != "kv_first":
            if rule == "current" and kv > 0:
                check_parity(st.kvload, kv - 1)
                if st.kvload.done < kv:
                    break
            if t >= NQ:
                bar, c = st.qempty[t % NQ], t // NQ - 1
                check_parity(bar, c)
                if bar.done < c + 1:
                    break
            st.rec[t % NQ] = (kv, m + ng >= T)
            yield ("async", ("q", t))
            t, m = t + 1, m + 1
        if rule == "per_tile_o":
            for j in range(t_first - ng, t_first):
                if j >= 0:
                    yield ("wait", st.ofull[j % ng], j // ng)
        elif kv > 0:
            yield ("wait", st.kvfree, kv - 1)
        for g, kvt in st.inflight.items():
            assert kvt >= kv, f"K/V load {kv} issued while group {g} still computes with load {kvt}"
        st.kv_in_buffer = kv
        yield ("async", ("kv", kv))
        kv_loads += 1
        for _ in range(max(0, ng - T)):
            st.kvfree.arrive(kv)
        while m < T:
            if t >= NQ:
                yield ("wait", st.qempty[t % NQ], t // NQ - 1)
            st.rec[t % NQ] = (kv, m + ng >= T)
            yield ("async", ("q", t))
            t, m = t + 1, m + 1
    for _ in range(ng):
        if t >= NQ:
            yield ("wait", st.qempty[t % NQ], t // NQ - 1)
        st.rec[t % NQ] = END
        st.qfull[t % NQ].arrive(t // NQ)
        t += 1


def group(st, g):
    ng, it, k, kv_seen = st.ng, g, 0, -1
    while True:
        yield ("wait", st.qfull[it % NQ], it // NQ)
        rec = st.rec[it % NQ]
        if rec is END:
            return
        kv, last = rec
        if it >= ng:  # at the LayerNorm exchange: the group's previous tile's buffer is free
            st.qempty[(it - ng) % NQ].arrive((it - ng) // NQ)
        if kv != kv_seen:
            yield ("wait", st.kvload, kv)
            kv_seen = kv
        assert st.kv_in_buffer == kv, f"group {g} tile {it}: K/V buffer holds load {st.kv_in_buffer}, not {kv}"
        st.inflight[g] = kv
        yield ("async", ("o", g, k, kv if last else None))
        yield ("wait", st.ofull[g], k)
        it, k = it + ng, k + 1


def run(batches, ng, seed, rule="current"):
    rng = random.Random(seed)
    st = State(ng)
    procs = {"p": producer(st, batches, rule)}
    for g in range(ng):
        procs[f"g{g}"] = group(st, g)
    waiting = {}        # name -> (bar, c)
    events = []         # pending asynchronous completions

    def step(name):
        try:
            req = procs[name].send(None)
        except StopIteration:
            del procs[name]
            return
        if req[0] == "wait":
            _, bar, c = req
            check_parity(bar, c)
            if bar.done < c + 1:
                waiting[name] = (bar, c)
        elif req[0] == "async":
            events.append(req[1])

    for _ in range(200000):
        if not procs and not events:
            return
        ready = [n for n in procs if n not in waiting]
        choices = [("proc", n) for n in ready] + [("event", i) for i in range(len(events))]
        if not choices:
            raise Violation("deadlock: " + ", ".join(f"{n} waits {b.name} #{c}" for n, (b, c) in waiting.items()))
        kind, x = rng.choice(choices)
        if kind == "proc":
            step(x)
        else:
            ev = events.pop(x)
            if ev[0] == "q":
                st.qfull[ev[1] % NQ].arrive(ev[1] // NQ)
            elif ev[0] == "kv":
                st.kvload.arrive(ev[1])
            else:
                _, g, k, kv_last = ev
                st.ofull[g].arrive(k)
                st.inflight.pop(g, None)
                if kv_last is not None:
                    st.kvfree.arrive(kv_last)
        for n, (bar, c) in list(waiting.items()):
            check_parity(bar, c)
            if bar.done >= c + 1:
                del waiting[n]
    raise Violation("did not finish")


def _batches(rng):
    n = rng.randint(1, 24)
    return [rng.choice([0, 0, 1, 1, 2, 3, 4, 5, 8]) for _ in range(n)]


@pytest.mark.parametrize("rule", ["current", "kv_first"])
@pytest.mark.parametrize("ng", [1, 2])
def test_protocol_random_schedules(ng, rule):
    """The kernel's rule (a batch's first tiles go out early once the previous
    K/V load has landed), and the simpler one (every tile after the K/V load)."""
    rng = random.Random(1234 + ng)
    for case in range(400):
        run(_batches(rng), ng, seed=case, rule=rule)


@pytest.mark.parametrize("rule", ["per_tile_o", "early_unchecked"])
def test_protocol_catches_broken_rules(rule):
    """Two rules that are wrong: waiting at a batch switch on each group's
    per-tile O barrier for the parity of its last tile (reads a phase two
    behind as done); and issuing a batch's first tiles before the previous K/V
    load has landed (a group that had no tile in that batch then waits for the
    new load two phases ahead of the K/V barrier)."""
    rng = random.Random(99)
    caught = 0
    for case in range(400):
        try:
            run(_batches(rng), 2, seed=case, rule=rule)
        except (Violation, AssertionError):
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------- the cluster exchanges
def exchange_group(cta, g, ng, nslot, tiles, X1, X2, slots1, slots2, H):
    """One compute group of one CTA: per tile, push its LayerNorm partial to
    slot it % nslot of every CTA (a send completes transaction bytes on that
    CTA's barrier), wait for all H partials, read them; later the same for the
    RMSNorm partial, which the kernel sends only after the tile's O (itself
    after the LayerNorm exchange)."""
    for it in range(g, tiles, ng):
        s = it % nslot
        for X, slots in ((X1, slots1), (X2, slots2)):
            for c in range(H):
                prev = slots[c][s][cta]
                assert prev is None or prev[1], f"CTA {c} slot {s}: partial of tile {prev[0]} overwritten unread"
                X[c][s].arrive(it // nslot)
                slots[c][s][cta] = [it, False]
            yield ("wait", X[cta][s], it // nslot)
            for p in range(H):
                entry = slots[cta][s][p]
                assert entry[0] == it, f"CTA {cta} tile {it} read tile {entry[0]}'s partial"
                entry[1] = True


def run_exchanges(H, ng, nslot, tiles, seed):
    rng = random.Random(seed)
    X1 = [[Bar(f"x1[{c}][{s}]", count=H) for s in range(nslot)] for c in range(H)]
    X2 = [[Bar(f"x2[{c}][{s}]", count=H) for s in range(nslot)] for c in range(H)]
    slots1 = [[[None] * H for _ in range(nslot)] for _ in range(H)]
    slots2 = [[[None] * H for _ in range(nslot)] for _ in range(H)]
    procs = {(c, g): exchange_group(c, g, ng, nslot, tiles, X1, X2, slots1, slots2, H)
             for c in range(H) for g in range(ng)}
    waiting = {}
    for _ in range(200000):
        if not procs:
            return
        ready = [n for n in procs if n not in waiting]
        if not ready:
            raise Violation("deadlock in the exchanges")
        n = rng.choice(ready)
        try:
            _, bar, c = procs[n].send(None)
            check_parity(bar, c)
            if bar.done < c + 1:
                waiting[n] = (bar, c)
        except StopIteration:
            del procs[n]
        for w, (bar, c) in list(waiting.items()):
            check_parity(bar, c)
            if bar.done >= c + 1:
                del waiting[w]
    raise Violation("did not finish")


@pytest.mark.parametrize("H,ng", [(2, 2), (4, 2), (3, 1), (8, 1)])
def test_exchange_slots_one_per_group(H, ng):
    """One exchange slot per group (tile it uses slot it mod NG) is never
    overwritten before it is read, and every send lands in its phase."""
    for seed in range(150):
        run_exchanges(H, ng, ng, tiles=9, seed=seed)


def test_exchange_model_catches_shared_slot():
    """Two groups sharing one slot (tiles of both groups on slot 0) overwrite
    partials before they are read or send into the wrong phase."""
    caught = 0
    for seed in range(150):
        try:
            run_exchanges(4, 2, 1, tiles=9, seed=seed)
        except (Violation, AssertionError):
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------- the batch ring
class TxBar(Bar):
    """An mbarrier that also counts transaction bytes: a phase completes once
    its arrivals are all in and its expected bytes have all landed (in either
    order)."""

    def __init__(self, name, count=1):
        super().__init__(name, count)
        self.tx = 0

    def arrive_expect(self, phase, nbytes):
        assert self.done == phase, f"{self.name}: re-arm for phase {phase} while at phase {self.done}"
        self.tx += nbytes
        self.arrivals += 1
        self._complete()

    def complete_tx(self, phase, nbytes):
        assert self.done == phase, f"{self.name}: bytes for phase {phase} landed at phase {self.done}"
        self.tx -= nbytes
        self._complete()

    def _complete(self):
        if self.arrivals == self.count and self.tx == 0:
            self.done += 1
            self.arrivals = 0


def ring_cta(rank, H, nb, entries, bfull, bempty, ring, seen, check_empty=True, rearm=True):
    """One CTA's producer, in the kernel's order.  Rank 0 publishes entry k
    (the batch from the counter; the last entry is the end mark) with a 4-byte
    remote write into slot k % nb of every CTA's ring, counted on that CTA's
    bfull[slot], after waiting on bempty[slot] for every CTA to have read entry
    k - nb.  Every CTA waits for entry k on bfull, reads it, re-arms bfull for
    entry k + nb (one arrival expecting 4 bytes), then arrives on rank 0's
    bempty; rank 0 then publishes entry k + 1 (so it runs one entry ahead of
    the batch it works on).  A CTA stops after reading the end mark."""
    def publish(k):
        s = k % nb
        if k >= nb and check_empty:
            yield ("wait", bempty[s], k // nb - 1)
        for c in range(H):
            prev = ring[c][s]
            assert prev is None or prev[1], f"ring of CTA {c} slot {s}: entry {prev[0]} overwritten unread"
            ring[c][s] = [k, False]
            bfull[c][s].complete_tx(k // nb, 4)

    if rank == 0:
        yield from publish(0)
    for k in range(entries):
        s = k % nb
        yield ("wait", bfull[rank][s], k // nb)
        assert ring[rank][s][0] == k, f"CTA {rank} read entry {ring[rank][s][0]} for {k}"
        ring[rank][s][1] = True
        seen[rank].append(k)
        if rearm:
            bfull[rank][s].arrive_expect(k // nb + 1, 4)
        bempty[s].arrive(k // nb)
        if k == entries - 1:  # the end mark
            return
        if rank == 0:
            yield from publish(k + 1)


def run_ring(H, nb, entries, seed, check_empty=True, rearm=True):
    rng = random.Random(seed)
    bfull = [[TxBar(f"bfull[{c}][{s}]") for s in range(nb)] for c in range(H)]
    for c in range(H):  # set-up: every slot armed for its first entry
        for s in range(nb):
            bfull[c][s].arrive_expect(0, 4)
    bempty = [Bar(f"bempty[{s}]", count=H) for s in range(nb)]
    ring = [[None] * nb for _ in range(H)]
    seen = [[] for _ in range(H)]
    procs = {c: ring_cta(c, H, nb, entries, bfull, bempty, ring, seen, check_empty, rearm) for c in range(H)}
    waiting = {}
    for _ in range(200000):
        if not procs:
            assert all(s == list(range(entries)) for s in seen)
            return
        ready = [n for n in procs if n not in waiting]
        if not ready:
            raise Violation("deadlock in the batch ring")
        n = rng.choice(ready)
        try:
            _, bar, c = procs[n].send(None)
            check_parity(bar, c)
            if bar.done < c + 1:
                waiting[n] = (bar, c)
        except StopIteration:
            del procs[n]
        for w, (bar, c) in list(waiting.items()):
            check_parity(bar, c)
            if bar.done >= c + 1:
                del waiting[w]
    raise Violation("did not finish")


@pytest.mark.parametrize("H", [1, 2, 4, 8])
def test_batch_ring(H):
    """Every CTA sees every entry, in order; no entry is overwritten unread."""
    for seed in range(150):
        run_ring(H, 4, entries=23, seed=seed)


def test_batch_ring_model_catches_missing_empty_wait():
    caught = 0
    for seed in range(150):
        try:
            run_ring(4, 2, entries=23, seed=seed, check_empty=False)
        except (Violation, AssertionError):
            caught += 1
    assert caught > 0


def test_batch_ring_model_catches_missing_rearm():
    """Without the re-arm, an entry's bytes land in a phase with no arrival
    pending: the phase never completes."""
    for seed in range(20):
        with pytest.raises(Violation):
            run_ring(2, 2, entries=9, seed=seed, rearm=False)
