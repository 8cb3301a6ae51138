"""CPU model of the forward kernel's barrier protocol, role by role (no GPU).

"4.3 FlashAttention 2 & 3", section "A from-scratch model of the
producer/consumer pipeline", checks a warp-specialised pipeline by modelling
its producer and consumers.  This file models the forward kernel's own roles
-- the load warp, the MMA-issuing warp and the two query tiles' softmax warps
-- with every mbarrier wait and arrival in the order the kernel performs them,
for both issue orders the kernel uses:
  * coupled (bf16, d = 128): P is written over S in TMEM, so S_t(j+1) is issued
    after P_t(j).V; causal units may let tile 0 skip the pair's last block;
  * decoupled (FP8: P in shared memory; bf16 d = 64: P in TMEM columns of its
    own): S_t(j+1) is issued once the softmax has read S_t(j) (s_free), ahead
    of P_t(j).V, and the softmax refills its P buffer only after the previous
    P.V completed (p_free).
Units are random sequences of key-block counts (split-KV's empty ranges
included).  Completions (TMA copies, tcgen05 commits) arrive as soon as they
are issued, which only removes delays and so cannot hide a deadlock.

Checked: every role finishes (no wait that never completes); every S product
lands in a TMEM buffer whose previous S the softmax has already read; every
P.V reads the P it is meant to, and no P is overwritten before its P.V read
it; the K/V ring never refills a slot before its tile was consumed; every
product of a unit is issued before the unit's output is read; no S product
reads a Q tile the next unit's copy has replaced.  Mutations of
the protocol (a wait dropped, a wrong parity, a barrier shared by two P
buffers) must be caught.
"""
import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals complete a phase; a wait with parity P
    succeeds while the number of completed phases has the other parity."""

    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def ready(self, parity):
        return (self.done & 1) != parity


class Violation(Exception):
    pass


def simulate(units, decoupled, stages, mutate=None, seed=0):
    """Runs the roles over `units`, a list of (nblocks, skip0) per unit.
    Returns the roles still waiting (empty when all finished); raises
    Violation on a safety failure."""
    bars = {}

    def bar(name, count=1):
        return bars.setdefault(name, Bar(count))

    for s in range(stages):
        bar(("kv_full", s)), bar(("kv_empty", s))
    for t in range(2):
        for n in ("q_full", "q_empty", "s_full", "p_ready", "o_final", "s_free", "p_free"):
            bar((n, t))
    # Safety state: what each TMEM / shared buffer holds.
    ring = [None] * stages          # item index held by each ring slot
    q_buf = [None, None]            # unit whose Q tile t is in shared memory
    s_buf = [None, None]            # (unit, block) of the S product in tile t's S columns
    s_read = [None, None]           # last (unit, block) the softmax read from them
    p_buf = [None, None]            # (unit, block) of the P stored for tile t
    p_used = [None, None]           # last (unit, block) whose P.V read that P
    pv_done = [set(), set()]        # (unit, block) P.V issued per tile

    def load():
        item = 0
        for u, (J, _) in enumerate(units):
            if J == 0:
                continue
            for t in range(2):
                uq = sum(1 for v in units[:u] if v[0] > 0)
                if uq > 0 and mutate != "load_skips_q_empty":
                    yield ("q_empty", t), (uq - 1) & 1
                q_buf[t] = u
                bar(("q_full", t)).arrive()
            for j in range(J):
                for kv in range(2):
                    slot, ph = item % stages, (item // stages) & 1
                    if mutate != "load_skips_empty_wait":
                        yield ("kv_empty", slot), ph ^ 1
                    if ring[slot] is not None:
                        raise Violation(f"ring slot {slot} refilled while item {ring[slot]} is in use")
                    ring[slot] = item
                    bar(("kv_full", slot)).arrive()
                    item += 1

    def consume(item):
        slot = item % stages
        yield ("kv_full", slot), (item // stages) & 1
        if ring[slot] != item:
            raise Violation(f"item {item} not in slot {slot} (holds {ring[slot]})")

    def release(item):
        ring[item % stages] = None
        bar(("kv_empty", item % stages)).arrive()

    def mma():
        item, uit = 0, 0
        ns, npv = [0, 0], [0, 0]

        def s_product(u, t, j):
            if decoupled:
                if ns[t] > 0:
                    parity = (ns[t] - 1) & 1
                    if mutate == "mma_s_free_wrong_parity":
                        parity ^= 1
                    if mutate != "mma_skips_s_free":
                        yield ("s_free", t), parity
            if q_buf[t] != u:
                raise Violation(f"S of tile {t} unit {u} reads Q of unit {q_buf[t]}")
            if s_buf[t] is not None and s_read[t] != s_buf[t]:
                raise Violation(f"S of tile {t} overwritten before the softmax read {s_buf[t]}")
            if not decoupled and s_buf[t] is not None and s_buf[t] not in pv_done[t]:
                raise Violation(f"S/P columns of tile {t} overwritten before P.V of {s_buf[t]}")
            s_buf[t] = (u, j)
            ns[t] += 1
            bar(("s_full", t)).arrive()

        def pv_product(u, t, j):
            parity = npv[t] & 1
            yield ("p_ready", t), parity
            if p_buf[t] != (u, j):
                raise Violation(f"P.V of tile {t} block {(u, j)} reads P of {p_buf[t]}")
            p_used[t] = (u, j)
            pv_done[t].add((u, j))
            npv[t] += 1
            if decoupled:
                bar(("p_free", t)).arrive()

        for u, (J, skip0) in enumerate(units):
            if J == 0:
                continue
            yield ("q_full", 0), uit & 1
            yield ("q_full", 1), uit & 1
            base = item
            item += 2 * J
            if decoupled:
                yield from consume(base)
                yield from s_product(u, 0, 0)
                yield from s_product(u, 1, 0)
                release(base)
                if J == 1:
                    bar(("q_empty", 0)).arrive(), bar(("q_empty", 1)).arrive()
                for j in range(J):
                    iv, ik = base + 2 * j + 1, base + 2 * j + 2
                    if j + 1 < J:
                        yield from consume(ik)
                        yield from s_product(u, 0, j + 1)
                        yield from s_product(u, 1, j + 1)
                        release(ik)
                        if j + 2 == J:
                            bar(("q_empty", 0)).arrive(), bar(("q_empty", 1)).arrive()
                    yield from consume(iv)
                    yield from pv_product(u, 0, j)
                    if j == J - 1:
                        bar(("o_final", 0)).arrive()
                    yield from pv_product(u, 1, j)
                    release(iv)
                    if j == J - 1:
                        bar(("o_final", 1)).arrive()
            else:
                J0 = J - 1 if skip0 else J
                yield from consume(base)
                yield from s_product(u, 0, 0)
                yield from s_product(u, 1, 0)
                release(base)
                if J == 1:
                    bar(("q_empty", 0)).arrive(), bar(("q_empty", 1)).arrive()
                for j in range(J):
                    iv, ik = base + 2 * j + 1, base + 2 * j + 2
                    yield from consume(iv)
                    if j < J0:
                        yield from pv_product(u, 0, j)
                        if j == J0 - 1:
                            bar(("o_final", 0)).arrive()
                    if j + 1 < J:
                        yield from consume(ik)
                        if j + 1 < J0:
                            yield from s_product(u, 0, j + 1)
                    yield from pv_product(u, 1, j)
                    release(iv)
                    if j == J - 1:
                        bar(("o_final", 1)).arrive()
                    if j + 1 < J:
                        yield from s_product(u, 1, j + 1)
                        release(ik)
                        if j + 2 == J:
                            bar(("q_empty", 0)).arrive(), bar(("q_empty", 1)).arrive()
            uit += 1

    def softmax(t):
        sit, np_, uit = 0, 0, 0
        for u, (J, skip0) in enumerate(units):
            if J == 0:
                continue   # an empty key range: the softmax writes its empty result
            nb = J - 1 if (skip0 and t == 0 and not decoupled) else J
            for j in range(nb):
                yield ("s_full", t), sit & 1
                sit += 1
                if s_buf[t] != (u, j):
                    raise Violation(f"softmax {t} expected S of {(u, j)}, TMEM holds {s_buf[t]}")
                s_read[t] = (u, j)
                if decoupled:
                    bar(("s_free", t)).arrive()
                    if np_ > 0 and mutate != "softmax_skips_p_free":
                        yield ("p_free", t), (np_ - 1) & 1
                # P of this block replaces the tile's previous P.
                if p_buf[t] is not None and p_used[t] != p_buf[t]:
                    raise Violation(f"P of tile {t} block {p_buf[t]} overwritten before its P.V")
                p_buf[t] = (u, j)
                bar(("p_ready", t)).arrive()
                np_ += 1
            yield ("o_final", t), uit & 1
            missing = [j for j in range(nb) if (u, j) not in pv_done[t]]
            if missing:
                raise Violation(f"tile {t} reads O of unit {u} before P.V of blocks {missing}")
            uit += 1

    roles = {"load": load(), "mma": mma(), "softmax0": softmax(0), "softmax1": softmax(1)}
    waiting = dict.fromkeys(roles)
    live = set(roles)
    rng = random.Random(seed)
    while live:
        moved = False
        order = sorted(live)
        rng.shuffle(order)   # any interleaving of the roles' progress
        for r in order:
            w = waiting[r]
            if w is not None and not bars[w[0]].ready(w[1]):
                continue
            try:
                waiting[r] = next(roles[r])
            except StopIteration:
                live.discard(r)
            moved = True
        if not moved:
            break
    return {r: waiting[r] for r in live}


def random_units(rng, causal):
    units = []
    for _ in range(rng.randint(1, 6)):
        J = rng.choice([0, 1, 1, 2, 3, 5, 8, 13])
        units.append((J, causal and J >= 2 and rng.random() < 0.5))
    return units


@pytest.mark.parametrize("decoupled,stages", [(False, 4), (True, 8), (True, 4)])
def test_protocol_completes_and_is_safe(decoupled, stages):
    rng = random.Random(1000 + stages + 10 * decoupled)
    for case in range(150):
        units = random_units(rng, causal=not decoupled)
        stuck = simulate(units, decoupled, stages, seed=case)
        assert not stuck, (units, stuck)


@pytest.mark.parametrize("mutation,decoupled", [
    ("mma_skips_s_free", True),
    ("mma_s_free_wrong_parity", True),
    ("softmax_skips_p_free", True),
    ("load_skips_empty_wait", True),
    ("load_skips_empty_wait", False),
    ("load_skips_q_empty", False),
    ("load_skips_q_empty", True),
])
def test_protocol_mutations_are_caught(mutation, decoupled):
    """Each mutation must end in a safety violation or a role that never
    finishes, for some unit sequence."""
    rng = random.Random(7)
    caught = False
    for case in range(200):
        units = random_units(rng, causal=not decoupled)
        try:
            stuck = simulate(units, decoupled, 4 if not decoupled else 8, mutate=mutation, seed=case)
        except Violation:
            caught = True
            break
        if stuck:
            caught = True
            break
    assert caught, mutation


def test_two_p_buffers_on_one_barrier_deadlock():
    """With two P buffers per tile the softmax may store P(j+1) before the MMA
    warp has waited for P(j); a single P-ready barrier then completes two
    phases before the wait and the MMA warp never sees the first.  The model
    (one barrier, the softmax refilling a buffer only after the P.V two blocks
    back) reproduces that hang."""
    b = Bar(1)
    b.arrive()           # P(0) stored
    b.arrive()           # P(1) stored into the other buffer
    assert not b.ready(0)   # the wait for P(0) (parity 0) can no longer succeed
