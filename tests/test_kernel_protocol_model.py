"""CPU model of the forward kernel's barrier protocol, role by role (no GPU).

"4.3 FlashAttention 2 & 3", section "A from-scratch model of the
producer/consumer pipeline", checks a warp-specialised pipeline by modelling
its producer and consumers.  This file models the forward kernel's own roles
-- the load warp, the MMA-issuing warp and the two query tiles' softmax warps
-- with every mbarrier wait and arrival in the order the kernel performs them,
for the three issue orders the kernel uses:
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
    and the rest of P follows (p_ready: the remaining P.V steps, p_free).
The MMA warp's products and commits go into an in-order tensor pipe that a
role of its own executes at any later point: a product reads and writes its
buffers when it runs, and a commit arrives once everything issued before it
has run.  Copies land as soon as they are issued, which only removes delays.
Every role runs at a random speed, so that one can run far ahead of another.
Softmax blocks are retaken at random (the reference moves and O is rescaled):
the coupled order rescales right after the block's S arrived, the decoupled
order after the previous P.V (p_free), the split order before signalling P's
last keys (after p_free) or after it (after pt_done).
Units are random sequences of key-block counts (split-KV's empty ranges
included).

Checked at every step: every role finishes (no wait that never completes); no
S product overwrites an S the softmax has not read or a P whose P.V has not
run; every P.V reads the P of its block; no P is refilled before its P.V
ran; the K/V ring never refills a slot before its tile was consumed; no
product reads a Q tile the next unit's copy has replaced; the softmax reads S
only once all of it is the block's; O is rescaled only once every product
accumulating into it has run, and read only once all of the unit's have.
Mutations of the protocol (a wait dropped, a wrong parity, a product issued
out of order, a barrier shared by two P buffers) must be caught.
"""
import random
from collections import deque

import pytest

ORDERS = ("coupled", "decoupled", "split")


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


def run_roles(roles, bars, seed):
    """Advances the roles in a random order until all finish or none can move.
    A role yields either (barrier, parity) or a predicate to wait on.  Each
    role gets a random speed (the chance that it takes a ready step in a
    sweep); the run ends when no role is ready.  Returns the roles still
    waiting."""
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


def simulate(units, order, stages, mutate=None, seed=0):
    """Runs the roles of `order` over `units`, a list of (nblocks, skip0) per
    unit.  Returns the roles still waiting (empty when all finished); raises
    Violation on a safety failure."""
    assert order in ORDERS
    split, coupled = order == "split", order == "coupled"
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
    # TMEM contents of S_t's columns: "main" (coupled and decoupled: all of
    # them) and, in the split order, "tail"; a region holds ("S", unit, block)
    # or ("P", unit, block).
    s_reg = [{"main": None, "tail": None}, {"main": None, "tail": None}]
    s_read = [None, None]            # last (unit, block) whose S the softmax read
    p_buf = [None, None]             # P outside S (FP8: shared memory; split: own columns)
    ran = [set(), set()]             # ("tail" | "main", unit, block) P.V steps that ran
    pipe = deque()
    mma_done = [False]
    retake_rng = random.Random(seed + 7)

    # ------------------------------------------------------------ load warp
    def load():
        item, uq = 0, 0
        for u, (J, _) in enumerate(units):
            if J == 0:
                continue
            for t in range(2):
                if uq > 0 and mutate != "load_skips_q_empty":
                    yield ("q_empty", t), (uq - 1) & 1
                q_buf[t] = u
                bar(("q_full", t)).arrive()
            uq += 1
            for j in range(J):
                for kv in range(2):
                    slot, ph = item % stages, (item // stages) & 1
                    if mutate != "load_skips_empty_wait":
                        yield ("kv_empty", slot), ph ^ 1
                        if ring[slot] is not None:
                            raise Violation(f"ring slot {slot} refilled while item {ring[slot]} "
                                            f"is in use")
                    ring[slot] = item
                    bar(("kv_full", slot)).arrive()
                    item += 1

    # ---------------------------------------- products, run by the tensor pipe
    def check_ring(item, what):
        if ring[item % stages] != item:
            raise Violation(f"{what} reads ring item {ring[item % stages]}, not {item}")

    def run_s(t, u, j, kitem, reg):
        check_ring(kitem, f"S of tile {t} {(u, j)}")
        if q_buf[t] != u:
            raise Violation(f"S of tile {t} unit {u} reads Q of unit {q_buf[t]}")
        held = s_reg[t][reg]
        if held is not None:
            kind, key = held[0], held[1:]
            if kind == "S" and s_read[t] != key:
                raise Violation(f"S ({reg}) of tile {t} overwritten before the softmax read {key}")
            if kind == "P" and ("tail" if split else "main", *key) not in ran[t]:
                raise Violation(f"S ({reg}) of tile {t} overwrites P of {key} before its P.V")
        s_reg[t][reg] = ("S", u, j)

    def run_pv(t, u, j, vitem, part):
        check_ring(vitem, f"P.V of tile {t} {(u, j)}")
        if coupled:
            held = s_reg[t]["main"]
        elif split and part == "tail":
            held = s_reg[t]["tail"]
        else:
            held = ("P", *p_buf[t]) if p_buf[t] is not None else None
        if held != ("P", u, j):
            raise Violation(f"P.V ({part}) of tile {t} block {(u, j)} reads {held}")
        ran[t].add((part, u, j))

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

    # ------------------------------------------------------------ MMA warp
    def mma():
        item, uit, npv = 0, 0, 0
        ns = [0, 0]
        pr = [0, 0]

        def s_after_free(t, u, j, kitem):
            if ns[t] > 0 and mutate != "mma_skips_s_free":
                parity = (ns[t] - 1) & 1
                if mutate == "mma_s_free_wrong_parity":
                    parity ^= 1
                yield ("s_free", t), parity
            ns[t] += 1
            issue(run_s, t, u, j, kitem, "main")

        def s0_coupled(u, j, kitem, J0):
            if j < J0:
                issue(run_s, 0, u, j, kitem, "main")
                commit(("s_full", 0))

        for u, (J, skip0) in enumerate(units):
            if J == 0:
                continue
            yield ("q_full", 0), uit & 1
            yield ("q_full", 1), uit & 1
            base = item
            item += 2 * J
            yield ("kv_full", base % stages), (base // stages) & 1
            if coupled:
                J0 = J - 1 if skip0 else J
                for t in range(2):
                    issue(run_s, t, u, 0, base, "main")
                    commit(("s_full", t))
                issue(run_release, base % stages)
                if J == 1:
                    commit(("q_empty", 0)), commit(("q_empty", 1))
                for j in range(J):
                    iv, ik = base + 2 * j + 1, base + 2 * j + 2
                    yield ("kv_full", iv % stages), (iv // stages) & 1
                    if j + 1 < J and mutate == "mma_s_before_pv":
                        yield ("kv_full", ik % stages), (ik // stages) & 1
                        s0_coupled(u, j + 1, ik, J0)
                    if j < J0:
                        yield ("p_ready", 0), pr[0] & 1
                        pr[0] += 1
                        issue(run_pv, 0, u, j, iv, "main")
                        if j == J0 - 1:
                            commit(("o_final", 0))
                    if j + 1 < J and mutate != "mma_s_before_pv":
                        yield ("kv_full", ik % stages), (ik // stages) & 1
                        s0_coupled(u, j + 1, ik, J0)
                    yield ("p_ready", 1), pr[1] & 1
                    pr[1] += 1
                    issue(run_pv, 1, u, j, iv, "main")
                    issue(run_release, iv % stages)
                    if j == J - 1:
                        commit(("o_final", 1))
                    if j + 1 < J:
                        issue(run_s, 1, u, j + 1, ik, "main")
                        commit(("s_full", 1))
                        issue(run_release, ik % stages)
                        if j + 2 == J:
                            commit(("q_empty", 0)), commit(("q_empty", 1))
            else:
                for t in range(2):
                    yield from s_after_free(t, u, 0, base)
                    if split:
                        # The previous unit's last P.V steps, already issued,
                        # read P's last keys before this overwrites them.
                        issue(run_s, t, u, 0, base, "tail")
                    commit(("s_full", t))
                issue(run_release, base % stages)
                if J == 1:
                    commit(("q_empty", 0)), commit(("q_empty", 1))
                for j in range(J):
                    iv, ik = base + 2 * j + 1, base + 2 * j + 2
                    nxt = j + 1 < J
                    if nxt:
                        yield ("kv_full", ik % stages), (ik // stages) & 1
                        for t in range(2):
                            yield from s_after_free(t, u, j + 1, ik)
                            if not split:
                                commit(("s_full", t))
                        if not split:
                            issue(run_release, ik % stages)
                            if j + 2 == J:
                                commit(("q_empty", 0)), commit(("q_empty", 1))
                    yield ("kv_full", iv % stages), (iv // stages) & 1
                    if split:
                        for t in range(2):
                            yield ("p_tail", t), npv & 1
                            if mutate == "mma_tail_before_pv" and nxt:
                                issue(run_s, t, u, j + 1, ik, "tail")
                                commit(("s_full", t))
                            issue(run_pv, t, u, j, iv, "tail")
                            commit(("pt_done", t))
                            if nxt and mutate != "mma_tail_before_pv":
                                issue(run_s, t, u, j + 1, ik, "tail")
                                commit(("s_full", t))
                    for t in range(2):
                        yield ("p_ready", t), npv & 1
                        issue(run_pv, t, u, j, iv, "main")
                        commit(("p_free", t))
                        if j == J - 1:
                            commit(("o_final", t))
                    issue(run_release, iv % stages)
                    if split and nxt:
                        issue(run_release, ik % stages)
                        if j + 2 == J:
                            commit(("q_empty", 0)), commit(("q_empty", 1))
                    npv += 1
            uit += 1
        mma_done[0] = True

    # ------------------------------------------------------------ softmax
    def rescale(t, u, j, steps):
        for step in steps:
            if step not in ran[t]:
                raise Violation(f"O of tile {t} rescaled at {(u, j)} before P.V step {step} ran")

    def softmax(t):
        sit, np_, uit = 0, 0, 0
        for u, (J, skip0) in enumerate(units):
            if J == 0:
                continue
            nb = J - 1 if (coupled and skip0 and t == 0) else J
            earlier = []                 # P.V steps of this unit issued so far
            for j in range(nb):
                yield ("s_full", t), sit & 1
                sit += 1
                want = ("S", u, j)
                if s_reg[t]["main"] != want or (split and s_reg[t]["tail"] != want):
                    raise Violation(f"softmax {t} expected S of {(u, j)}, TMEM holds {s_reg[t]}")
                s_read[t] = (u, j)
                if coupled:
                    if j > 0 and retake_rng.random() < 0.15:
                        rescale(t, u, j, earlier)
                    s_reg[t]["main"] = ("P", u, j)       # P over S (already read)
                    bar(("p_ready", t)).arrive()
                    earlier.append(("main", u, j))
                    continue
                bar(("s_free", t)).arrive()
                pfree_seen = np_ == 0
                if j > 0 and retake_rng.random() < 0.15:
                    if not pfree_seen and mutate != "softmax_skips_p_free":
                        yield ("p_free", t), (np_ - 1) & 1
                        pfree_seen = True
                    rescale(t, u, j, earlier)
                if split:
                    s_reg[t]["tail"] = ("P", u, j)       # P's last keys over S's tail (read)
                    bar(("p_tail", t)).arrive()
                if not pfree_seen and mutate != "softmax_skips_p_free":
                    yield ("p_free", t), (np_ - 1) & 1
                if p_buf[t] is not None and ("main", *p_buf[t]) not in ran[t]:
                    raise Violation(f"P of tile {t} block {p_buf[t]} overwritten before its P.V")
                p_buf[t] = (u, j)
                if split and retake_rng.random() < 0.15:
                    if mutate != "softmax_skips_pt_done":
                        yield ("pt_done", t), np_ & 1
                    rescale(t, u, j, earlier + [("tail", u, j)])
                bar(("p_ready", t)).arrive()
                np_ += 1
                earlier += [("tail", u, j), ("main", u, j)] if split else [("main", u, j)]
            yield ("o_final", t), uit & 1
            missing = [s for s in earlier if s not in ran[t]]
            if missing:
                raise Violation(f"tile {t} reads O of unit {u} before P.V steps {missing}")
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


@pytest.mark.parametrize("order,stages", [("coupled", 4), ("decoupled", 8), ("decoupled", 4),
                                          ("split", 8), ("split", 4)])
def test_protocol_completes_and_is_safe(order, stages):
    rng = random.Random(1000 + stages + 10 * ORDERS.index(order))
    for case in range(150):
        units = random_units(rng, causal=order == "coupled")
        stuck = simulate(units, order, stages, seed=case)
        assert not stuck, (units, stuck)


@pytest.mark.parametrize("mutation,order", [
    ("load_skips_empty_wait", "coupled"),
    ("load_skips_q_empty", "coupled"),
    ("mma_s_before_pv", "coupled"),
    ("mma_skips_s_free", "decoupled"),
    ("mma_s_free_wrong_parity", "decoupled"),
    ("softmax_skips_p_free", "decoupled"),
    ("load_skips_empty_wait", "decoupled"),
    ("load_skips_q_empty", "decoupled"),
    ("mma_skips_s_free", "split"),
    ("mma_s_free_wrong_parity", "split"),
    ("softmax_skips_p_free", "split"),
    ("mma_tail_before_pv", "split"),
    ("softmax_skips_pt_done", "split"),
    ("load_skips_empty_wait", "split"),
    ("load_skips_q_empty", "split"),
])
def test_protocol_mutations_are_caught(mutation, order):
    """Each mutation must end in a safety violation or a role that never
    finishes, for some unit sequence."""
    rng = random.Random(7)
    stages = 4 if order == "coupled" else 8
    for case in range(300):
        units = random_units(rng, causal=order == "coupled")
        try:
            stuck = simulate(units, order, stages, mutate=mutation, seed=case)
        except Violation:
            return
        if stuck:
            return
    pytest.fail(f"{mutation} ({order}) was not caught")


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
