"""CPU model of the forward kernel's barrier protocol, role by role (no GPU).

"4.3 FlashAttention 2 & 3", section "A from-scratch model of the
producer/consumer pipeline", checks a warp-specialised pipeline by modelling
its producer and consumers.  This file models the forward kernel's own roles
-- the load warp, the MMA-issuing warp and the two query tiles' softmax warps
-- with every mbarrier wait and arrival in the order the kernel performs them,
for both issue orders the kernel uses:
  * coupled (bf16, d = 128): P is written over S in TMEM, so S_t(j+1) is issued
    after P_t(j).V; causal units may let tile 0 skip the pair's last block;
  * decoupled (FP8: P in shared memory): S_t(j+1) is issued once the softmax
    has read S_t(j) (s_free), ahead of P_t(j).V, and the softmax refills its
    P buffer only after the previous P.V completed (p_free);
  * split (bf16, d = 64): as decoupled, but P's last keys are stored over the
    tail columns of S, so S_t(j+1) is issued in two parts -- its main part
    after s_free, its tail only after the P.V steps that read P's last keys.
    The softmax stores and signals those last keys first (p_tail), the MMA
    warp then issues their P.V steps (commit: pt_done) and S's tail (s_full),
    and the rest of P follows (p_ready: the remaining P.V steps, p_free).  A
    retaken block rescales O: before signalling the last keys after waiting
    for the previous block's P.V (p_free), or after it once their P.V is done
    (pt_done).
Units are random sequences of key-block counts (split-KV's empty ranges
included).  Completions (TMA copies, tcgen05 commits) arrive as soon as they
are issued, which only removes delays and so cannot hide a deadlock.

Checked: every role finishes (no wait that never completes); every S product
lands in a TMEM buffer whose previous S the softmax has already read; every
P.V reads the P it is meant to, and no P is overwritten before its P.V read
it; the K/V ring never refills a slot before its tile was consumed; every
product of a unit is issued before the unit's output is read; no S product
reads a Q tile the next unit's copy has replaced; in the split order, no S
tail overwrites P's last keys before their P.V steps read them, the softmax
reads an S whose two parts are both of the block, and O is rescaled only
while no product accumulates into it.  Mutations of the
protocol (a wait dropped, a wrong parity, a barrier shared by two P buffers,
an S tail issued too early) must be caught.
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


def simulate(units, decoupled, stages, mutate=None, seed=0, split=False):
    """Runs the roles over `units`, a list of (nblocks, skip0) per unit.
    Returns the roles still waiting (empty when all finished); raises
    Violation on a safety failure."""
    if split:
        return simulate_split(units, stages, mutate, seed)
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


def run_roles(roles, bars, seed):
    """Advances the roles in a random order until all finish or none can move.
    A role yields either (barrier, parity) or a predicate to wait on.  Each
    role gets a random speed (the chance that it takes a ready step in a
    sweep), so that one role can run far ahead of another; the run ends when
    no role is ready."""
    waiting = dict.fromkeys(roles)
    live = set(roles)
    rng = random.Random(seed)
    speed = {r: rng.choice([0.05, 0.3, 1.0]) for r in sorted(roles)}
    while live:
        any_ready = False
        order = sorted(live)
        rng.shuffle(order)
        for r in order:
            w = waiting[r]
            if w is not None:
                ready = w() if callable(w) else bars[w[0]].ready(w[1])
                if not ready:
                    continue
            any_ready = True
            if rng.random() > speed[r]:
                continue
            try:
                waiting[r] = next(roles[r])
            except StopIteration:
                live.discard(r)
        if not any_ready:
            break
    return {r: waiting[r] for r in live}


def simulate_split(units, stages, mutate=None, seed=0):
    """The split order (bf16, d = 64): S in a main part and a tail part, P's
    last keys over the tail columns of S.  Unlike the two orders above, the
    MMA warp's products and commits go into an in-order tensor pipe that a
    role of its own executes at any later point, so a product reads and
    writes its buffers when it runs and a commit arrives once everything
    issued before it has run; the checks are made at execution."""
    from collections import deque
    bars = {}

    def bar(name, count=1):
        return bars.setdefault(name, Bar(count))

    for s in range(stages):
        bar(("kv_full", s)), bar(("kv_empty", s))
    for t in range(2):
        for n in ("q_full", "q_empty", "s_full", "p_ready", "p_tail", "pt_done", "o_final",
                  "s_free", "p_free"):
            bar((n, t))
    ring = [None] * stages
    q_buf = [None, None]
    s_main_buf = [None, None]   # (unit, block) of S's main columns
    s_tail_buf = [None, None]   # (unit, block) of S's tail columns, or ("P", unit, block)
    s_read = [None, None]
    p_main = [None, None]       # P in the tile's own columns
    p_main_used = [None, None]
    p_tail_used = [None, None]  # last (unit, block) whose P.V read P's last keys
    pv_done = [set(), set()]    # (unit, block) whose P.V main steps ran
    tail_done = [set(), set()]  # (unit, block) whose P.V steps over the last keys ran
    pipe = deque()
    redo_rng = random.Random(seed + 7)
    mma_done = [False]

    def load():
        item = 0
        for u, (J, _) in enumerate(units):
            if J == 0:
                continue
            for t in range(2):
                uq = sum(1 for v in units[:u] if v[0] > 0)
                if uq > 0:
                    yield ("q_empty", t), (uq - 1) & 1
                q_buf[t] = u
                bar(("q_full", t)).arrive()
            for j in range(J):
                for kv in range(2):
                    slot, ph = item % stages, (item // stages) & 1
                    yield ("kv_empty", slot), ph ^ 1
                    if ring[slot] is not None:
                        raise Violation(f"ring slot {slot} refilled while item {ring[slot]} is in use")
                    ring[slot] = item
                    bar(("kv_full", slot)).arrive()
                    item += 1

    # ------------------------------------------------ products, run by the pipe
    def run_s_main(u, t, j, kitem):
        if ring[kitem % stages] != kitem:
            raise Violation(f"S of tile {t} reads ring item {ring[kitem % stages]}, not {kitem}")
        if q_buf[t] != u:
            raise Violation(f"S of tile {t} unit {u} reads Q of unit {q_buf[t]}")
        if s_main_buf[t] is not None and s_read[t] != s_main_buf[t]:
            raise Violation(f"S of tile {t} overwritten before the softmax read {s_main_buf[t]}")
        s_main_buf[t] = (u, j)

    def run_s_tail(u, t, j, kitem):
        if ring[kitem % stages] != kitem:
            raise Violation(f"S tail of tile {t} reads ring item {ring[kitem % stages]}, not {kitem}")
        if q_buf[t] != u:
            raise Violation(f"S tail of tile {t} unit {u} reads Q of unit {q_buf[t]}")
        tail = s_tail_buf[t]
        if tail is not None and tail[0] == "P" and p_tail_used[t] != tail[1:]:
            raise Violation(f"S tail of tile {t} overwrites P of {tail[1:]} before its P.V read it")
        if tail is not None and tail[0] != "P" and s_read[t] != tail:
            raise Violation(f"S tail of tile {t} overwritten before the softmax read {tail}")
        s_tail_buf[t] = (u, j)

    def run_pv_tail(u, t, j, vitem):
        if ring[vitem % stages] != vitem:
            raise Violation(f"P.V of tile {t} reads ring item {ring[vitem % stages]}, not {vitem}")
        if s_tail_buf[t] != ("P", u, j):
            raise Violation(f"P.V of tile {t} block {(u, j)} reads P's last keys of {s_tail_buf[t]}")
        p_tail_used[t] = (u, j)
        tail_done[t].add((u, j))

    def run_pv_main(u, t, j, vitem):
        if ring[vitem % stages] != vitem:
            raise Violation(f"P.V of tile {t} reads ring item {ring[vitem % stages]}, not {vitem}")
        if p_main[t] != (u, j):
            raise Violation(f"P.V of tile {t} block {(u, j)} reads P of {p_main[t]}")
        p_main_used[t] = (u, j)
        pv_done[t].add((u, j))

    def run_release(slot):
        ring[slot] = None
        bar(("kv_empty", slot)).arrive()

    def tensor():
        while True:
            yield lambda: bool(pipe) or mma_done[0]
            if not pipe:
                return
            fn, args = pipe.popleft()
            fn(*args)

    def issue(fn, *args):
        pipe.append((fn, args))

    def commit(name):
        issue(lambda: bar(name).arrive())

    def mma():
        item, uit, npv = 0, 0, 0
        ns = [0, 0]

        def s_main(u, t, j, kitem):
            if ns[t] > 0 and mutate != "mma_skips_s_free":
                yield ("s_free", t), (ns[t] - 1) & 1
            ns[t] += 1
            issue(run_s_main, u, t, j, kitem)

        def s_tail(u, t, j, kitem):
            issue(run_s_tail, u, t, j, kitem)
            commit(("s_full", t))

        for u, (J, _) in enumerate(units):
            if J == 0:
                continue
            yield ("q_full", 0), uit & 1
            yield ("q_full", 1), uit & 1
            base = item
            item += 2 * J
            yield ("kv_full", base % stages), (base // stages) & 1
            for t in range(2):
                yield from s_main(u, t, 0, base)
                s_tail(u, t, 0, base)
            issue(run_release, base % stages)
            if J == 1:
                commit(("q_empty", 0)), commit(("q_empty", 1))
            for j in range(J):
                iv, ik = base + 2 * j + 1, base + 2 * j + 2
                nxt = j + 1 < J
                if nxt:
                    yield ("kv_full", ik % stages), (ik // stages) & 1
                    yield from s_main(u, 0, j + 1, ik)
                    yield from s_main(u, 1, j + 1, ik)
                yield ("kv_full", iv % stages), (iv // stages) & 1
                for t in range(2):
                    yield ("p_tail", t), npv & 1
                    if mutate == "mma_tail_before_pv" and nxt:
                        s_tail(u, t, j + 1, ik)
                    issue(run_pv_tail, u, t, j, iv)
                    commit(("pt_done", t))
                    if nxt and mutate != "mma_tail_before_pv":
                        s_tail(u, t, j + 1, ik)
                for t in range(2):
                    yield ("p_ready", t), npv & 1
                    issue(run_pv_main, u, t, j, iv)
                    commit(("p_free", t))
                    if j == J - 1:
                        commit(("o_final", t))
                issue(run_release, iv % stages)
                if nxt:
                    issue(run_release, ik % stages)
                    if j + 2 == J:
                        commit(("q_empty", 0)), commit(("q_empty", 1))
                npv += 1
            uit += 1
        mma_done[0] = True

    def rescale(t, u, j, done):
        """O_t is rescaled: every P.V step that accumulates into it so far must
        have run (`done` lists the steps issued before this point)."""
        for kind, key in done:
            if key not in (tail_done[t] if kind == "tail" else pv_done[t]):
                raise Violation(f"O of tile {t} rescaled at {(u, j)} while P.V {kind} {key} "
                                f"has not run")

    def softmax(t):
        sit, np_, uit = 0, 0, 0
        prev = None
        for u, (J, _) in enumerate(units):
            if J == 0:
                continue
            for j in range(J):
                yield ("s_full", t), sit & 1
                sit += 1
                if s_main_buf[t] != (u, j) or s_tail_buf[t] != (u, j):
                    raise Violation(f"softmax {t} expected S of {(u, j)}, TMEM holds "
                                    f"{s_main_buf[t]} / {s_tail_buf[t]}")
                s_read[t] = (u, j)
                bar(("s_free", t)).arrive()
                pfree_seen = np_ == 0
                # A retake found on the last keys: wait for the previous P.V,
                # then rescale (O holds the unit's earlier blocks only).
                if j > 0 and redo_rng.random() < 0.15:
                    if not pfree_seen and mutate != "softmax_skips_p_free":
                        yield ("p_free", t), (np_ - 1) & 1
                        pfree_seen = True
                    rescale(t, u, j, [("main", prev)])
                s_tail_buf[t] = ("P", u, j)   # P's last keys over S's tail (already read)
                bar(("p_tail", t)).arrive()
                if not pfree_seen and mutate != "softmax_skips_p_free":
                    yield ("p_free", t), (np_ - 1) & 1
                if p_main[t] is not None and p_main_used[t] != p_main[t]:
                    raise Violation(f"P of tile {t} block {p_main[t]} overwritten before its P.V")
                p_main[t] = (u, j)
                # A retake found on the whole block: O already takes P.V over
                # this block's last keys; wait for it (pt_done), then rescale.
                if redo_rng.random() < 0.15:
                    if mutate != "softmax_skips_pt_done":
                        yield ("pt_done", t), np_ & 1
                    steps = [("tail", (u, j))] + ([("main", prev)] if j > 0 else [])
                    rescale(t, u, j, steps)
                bar(("p_ready", t)).arrive()
                np_ += 1
                prev = (u, j)
            yield ("o_final", t), uit & 1
            missing = [j for j in range(J) if (u, j) not in pv_done[t]]
            if missing:
                raise Violation(f"tile {t} reads O of unit {u} before P.V of blocks {missing}")
            uit += 1

    roles = {"load": load(), "mma": mma(), "tensor": tensor(), "softmax0": softmax(0),
             "softmax1": softmax(1)}
    return run_roles(roles, bars, seed)


def random_units(rng, causal):
    units = []
    for _ in range(rng.randint(1, 6)):
        J = rng.choice([0, 1, 1, 2, 3, 5, 8, 13])
        units.append((J, causal and J >= 2 and rng.random() < 0.5))
    return units


@pytest.mark.parametrize("decoupled,stages,split", [(False, 4, False), (True, 8, False),
                                                     (True, 4, False), (True, 8, True),
                                                     (True, 4, True)])
def test_protocol_completes_and_is_safe(decoupled, stages, split):
    rng = random.Random(1000 + stages + 10 * decoupled + 100 * split)
    for case in range(150):
        units = random_units(rng, causal=not decoupled)
        stuck = simulate(units, decoupled, stages, seed=case, split=split)
        assert not stuck, (units, stuck)


@pytest.mark.parametrize("mutation,decoupled,split", [
    ("mma_skips_s_free", True, False),
    ("mma_s_free_wrong_parity", True, False),
    ("softmax_skips_p_free", True, False),
    ("load_skips_empty_wait", True, False),
    ("load_skips_empty_wait", False, False),
    ("load_skips_q_empty", False, False),
    ("load_skips_q_empty", True, False),
    ("mma_skips_s_free", True, True),
    ("softmax_skips_p_free", True, True),
    ("mma_tail_before_pv", True, True),
    ("softmax_skips_pt_done", True, True),
])
def test_protocol_mutations_are_caught(mutation, decoupled, split):
    """Each mutation must end in a safety violation or a role that never
    finishes, for some unit sequence."""
    rng = random.Random(7)
    caught = False
    for case in range(200):
        units = random_units(rng, causal=not decoupled)
        try:
            stuck = simulate(units, decoupled, 4 if not decoupled else 8, mutate=mutation, seed=case,
                             split=split)
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
