"""CPU model of the backward kernels' barrier protocols, role by role (no GPU).

The backward of "4.3 FlashAttention 2 & 3" (section "The backward pass:
recompute, and the one identity that makes it tile-able") runs here as two
warp-specialised kernels; like the forward's model (its section "A from-scratch
model of the producer/consumer pipeline"), this file models each kernel's own
roles with every mbarrier wait and arrival in the kernel's order:
  * dK/dV kernel (unit = KV head x 128-key block): the load warp puts K_j and V_j
    in fixed buffers (fix_full / fix_empty) and streams Q_i, dO_i through a
    ring; the MMA warp issues S^T = K Q^T and dP^T = V dO^T into TMEM, the
    element-wise warps write P^T over S^T (p_ready) and dS^T over dP^T
    (ds_ready), and the MMA warp issues dV += P^T dO and dK += dS^T Q, each
    next S^T / dP^T after the product that reads the columns it overwrites;
  * dQ kernel (unit = head x 128-query block): the element-wise warps put Q_i
    and dO_i in TMEM (fix_full) once the previous unit is done; the load warp
    streams K_j, V_j through a ring; S = Q K^T is issued once the element-wise
    warps have read the previous S (s_read), dP = dO V^T after the dQ product
    that reads the dS written over the previous dP (p_ready).
The MMA warp's products and commits go into an in-order tensor pipe that a
role of its own executes later (a product reads and writes its buffers when
it runs; a commit arrives once everything issued before it has run).  The
element-wise warps are two roles, each owning half of every TMEM region, so
a barrier completes only once both have arrived.  Every role runs at a
random speed.  Units are random sequences of block counts.

Checked: every role finishes; no product overwrites a TMEM region before its
content was read (by the element-wise warps, or by the product that consumes
it); every product reads the block it is meant to; the ring and the fixed
buffers are never refilled while a product still needs them; an output is
read only once all its products have run.  Mutations (a product issued early,
a wait dropped) must be caught.
"""
import random
from collections import deque

import pytest

from test_kernel_protocol_model import Bar, Violation, run_roles

EW = (0, 1)   # the two element-wise roles


def _pipe_roles(bars):
    pipe = deque()
    done = [False]

    def tensor():
        while True:
            yield lambda: bool(pipe) or done[0]
            if not pipe:
                return
            fn, args = pipe.popleft()
            fn(*args)

    def issue(fn, *args):
        pipe.append((fn, args))

    def commit(name):
        issue(lambda: bars[name].arrive())

    return tensor, issue, commit, done


def simulate_dkdv(units, stages, mutate=None, seed=0):
    """units: list of T (query blocks per key block, >= 1)."""
    bars = {}

    def bar(name, count=1):
        return bars.setdefault(name, Bar(count))

    for s in range(stages):
        bar(("full", s)), bar(("empty", s))
    for n in ("fix_full", "fix_empty", "s_full", "dp_full", "unit_done"):
        bar(n)
    bar("p_ready", len(EW)), bar("ds_ready", len(EW))
    tensor, issue, commit, mma_done = _pipe_roles(bars)

    ring = [None] * stages
    fix = [None]                     # unit whose K_j, V_j are in the fixed buffers
    s_reg = {h: None for h in EW}    # ("S" | "P", unit, t)
    dp_reg = {h: None for h in EW}   # ("dP" | "dS", unit, t)
    ran = set()                      # ("S" | "dP" | "dV" | "dK", unit, t)

    def load():
        item = 0
        for u, T in enumerate(units):
            if u > 0 and mutate != "load_skips_fix_empty":
                yield "fix_empty", (u - 1) & 1
            fix[0] = u
            bar("fix_full").arrive()
            for t in range(T):
                for w in range(2):   # Q_t, dO_t
                    slot = item % stages
                    if mutate != "load_skips_empty_wait":
                        yield ("empty", slot), ((item // stages) & 1) ^ 1
                    ring[slot] = (u, t, "Q" if w == 0 else "dO")
                    bar(("full", slot)).arrive()
                    item += 1

    def need(item, want, what):
        if ring[item % stages] != want:
            raise Violation(f"{what} reads ring slot holding {ring[item % stages]}, not {want}")

    def run_S(u, t, item):
        need(item, (u, t, "Q"), f"S^T {(u, t)}")
        if fix[0] != u:
            raise Violation(f"S^T {(u, t)} reads K of unit {fix[0]}")
        for h in EW:
            held = s_reg[h]
            if held is not None and (held[0] != "P" or ("dV", *held[1:]) not in ran):
                raise Violation(f"S^T {(u, t)} overwrites {held} before it was consumed")
            s_reg[h] = ("S", u, t)
        ran.add(("S", u, t))

    def run_dP(u, t, item):
        need(item, (u, t, "dO"), f"dP^T {(u, t)}")
        if fix[0] != u:
            raise Violation(f"dP^T {(u, t)} reads V of unit {fix[0]}")
        for h in EW:
            held = dp_reg[h]
            if held is not None and (held[0] != "dS" or ("dK", *held[1:]) not in ran):
                raise Violation(f"dP^T {(u, t)} overwrites {held} before it was consumed")
            dp_reg[h] = ("dP", u, t)
        ran.add(("dP", u, t))

    def run_dV(u, t, item):
        need(item, (u, t, "dO"), f"dV {(u, t)}")
        for h in EW:
            if s_reg[h] != ("P", u, t):
                raise Violation(f"dV {(u, t)} reads {s_reg[h]}")
        ran.add(("dV", u, t))

    def run_dK(u, t, item):
        need(item, (u, t, "Q"), f"dK {(u, t)}")
        for h in EW:
            if dp_reg[h] != ("dS", u, t):
                raise Violation(f"dK {(u, t)} reads {dp_reg[h]}")
        ran.add(("dK", u, t))

    def run_release(slot):
        ring[slot] = None
        bar(("empty", slot)).arrive()

    def run_fix_release(u):
        for t in range(units[u]):
            if ("S", u, t) not in ran or ("dP", u, t) not in ran:
                raise Violation(f"K/V of unit {u} released before its products ran")
        bar("fix_empty").arrive()

    def mma():
        item, gblk = 0, 0
        for u, T in enumerate(units):
            yield "fix_full", u & 1
            base = item
            item += 2 * T
            yield ("full", base % stages), (base // stages) & 1
            yield ("full", (base + 1) % stages), ((base + 1) // stages) & 1
            issue(run_S, u, 0, base)
            commit("s_full")
            issue(run_dP, u, 0, base + 1)
            commit("dp_full")
            for t in range(T):
                iq, io = base + 2 * t, base + 2 * t + 1
                more = t + 1 < T
                if more and mutate == "mma_s_before_dv":
                    yield ("full", (iq + 2) % stages), ((iq + 2) // stages) & 1
                    issue(run_S, u, t + 1, iq + 2)
                    commit("s_full")
                yield "p_ready", gblk & 1
                issue(run_dV, u, t, io)
                issue(run_release, io % stages)
                if more and mutate != "mma_s_before_dv":
                    yield ("full", (iq + 2) % stages), ((iq + 2) // stages) & 1
                    issue(run_S, u, t + 1, iq + 2)
                    commit("s_full")
                if more and mutate == "mma_dp_before_dk":
                    yield ("full", (io + 2) % stages), ((io + 2) // stages) & 1
                    issue(run_dP, u, t + 1, io + 2)
                    commit("dp_full")
                yield "ds_ready", gblk & 1
                issue(run_dK, u, t, iq)
                issue(run_release, iq % stages)
                if more and mutate != "mma_dp_before_dk":
                    yield ("full", (io + 2) % stages), ((io + 2) // stages) & 1
                    issue(run_dP, u, t + 1, io + 2)
                    commit("dp_full")
                gblk += 1
            commit("unit_done")
            issue(run_fix_release, u)
        mma_done[0] = True

    def ew(h):
        gblk = 0
        for u, T in enumerate(units):
            for t in range(T):
                yield "s_full", gblk & 1
                if s_reg[h] != ("S", u, t):
                    raise Violation(f"element-wise {h} expected S^T {(u, t)}, TMEM holds {s_reg[h]}")
                s_reg[h] = ("P", u, t)          # P^T over S^T (read)
                bar("p_ready").arrive()
                if mutate != "ew_skips_dp_full":
                    yield "dp_full", gblk & 1
                if dp_reg[h] != ("dP", u, t):
                    raise Violation(f"element-wise {h} expected dP^T {(u, t)}, TMEM holds {dp_reg[h]}")
                dp_reg[h] = ("dS", u, t)        # dS^T over dP^T (read)
                bar("ds_ready").arrive()
                gblk += 1
            yield "unit_done", u & 1
            missing = [(k, u, t) for t in range(T) for k in ("dV", "dK") if (k, u, t) not in ran]
            if missing:
                raise Violation(f"element-wise {h} reads dK/dV of unit {u} before {missing}")

    roles = {"load": load(), "mma": mma(), "tensor": tensor()}
    roles.update({f"ew{h}": ew(h) for h in EW})
    return run_roles(roles, bars, seed)


def simulate_dq(units, stages, mutate=None, seed=0):
    """units: list of J (key blocks per query block, >= 1)."""
    bars = {}

    def bar(name, count=1):
        return bars.setdefault(name, Bar(count))

    for s in range(stages):
        bar(("full", s)), bar(("empty", s))
    for n in ("s_full", "dp_full", "unit_done"):
        bar(n)
    bar("fix_full", len(EW)), bar("s_read", len(EW)), bar("p_ready", len(EW))
    tensor, issue, commit, mma_done = _pipe_roles(bars)

    ring = [None] * stages
    qdo = {h: None for h in EW}      # unit whose Q_i, dO_i rows this role put in TMEM
    s_reg = {h: None for h in EW}    # ("S", unit, j)
    s_read = {h: None for h in EW}
    dp_reg = {h: None for h in EW}   # ("dP" | "dS", unit, j)
    ran = set()                      # ("S" | "dP" | "dQ", unit, j)

    def load():
        item = 0
        for u, J in enumerate(units):
            for j in range(J):
                for w in range(2):   # K_j, V_j
                    slot = item % stages
                    if mutate != "load_skips_empty_wait":
                        yield ("empty", slot), ((item // stages) & 1) ^ 1
                    ring[slot] = (u, j, "K" if w == 0 else "V")
                    bar(("full", slot)).arrive()
                    item += 1

    def need(item, want, what):
        if ring[item % stages] != want:
            raise Violation(f"{what} reads ring slot holding {ring[item % stages]}, not {want}")

    def run_S(u, j, item):
        need(item, (u, j, "K"), f"S {(u, j)}")
        for h in EW:
            if qdo[h] != u:
                raise Violation(f"S {(u, j)} reads Q rows of unit {qdo[h]}")
            if s_reg[h] is not None and s_read[h] != s_reg[h]:
                raise Violation(f"S {(u, j)} overwrites {s_reg[h]} before it was read")
            s_reg[h] = ("S", u, j)
        ran.add(("S", u, j))

    def run_dP(u, j, item):
        need(item, (u, j, "V"), f"dP {(u, j)}")
        for h in EW:
            if qdo[h] != u:
                raise Violation(f"dP {(u, j)} reads dO rows of unit {qdo[h]}")
            held = dp_reg[h]
            if held is not None and (held[0] != "dS" or ("dQ", *held[1:]) not in ran):
                raise Violation(f"dP {(u, j)} overwrites {held} before it was consumed")
            dp_reg[h] = ("dP", u, j)
        ran.add(("dP", u, j))

    def run_dQ(u, j, item):
        need(item, (u, j, "K"), f"dQ {(u, j)}")
        for h in EW:
            if dp_reg[h] != ("dS", u, j):
                raise Violation(f"dQ {(u, j)} reads {dp_reg[h]}")
        ran.add(("dQ", u, j))

    def run_release(slot):
        ring[slot] = None
        bar(("empty", slot)).arrive()

    def mma():
        item, gblk = 0, 0
        for u, J in enumerate(units):
            yield "fix_full", u & 1
            base = item
            item += 2 * J
            yield ("full", base % stages), (base // stages) & 1
            yield ("full", (base + 1) % stages), ((base + 1) // stages) & 1
            issue(run_S, u, 0, base)
            commit("s_full")
            issue(run_dP, u, 0, base + 1)
            commit("dp_full")
            issue(run_release, (base + 1) % stages)
            for j in range(J):
                ik = base + 2 * j
                more = j + 1 < J
                if more:
                    if mutate != "mma_skips_s_read":
                        yield "s_read", gblk & 1
                    yield ("full", (ik + 2) % stages), ((ik + 2) // stages) & 1
                    issue(run_S, u, j + 1, ik + 2)
                    commit("s_full")
                if more and mutate == "mma_dp_before_dq":
                    yield ("full", (ik + 3) % stages), ((ik + 3) // stages) & 1
                    issue(run_dP, u, j + 1, ik + 3)
                    commit("dp_full")
                    issue(run_release, (ik + 3) % stages)
                yield "p_ready", gblk & 1
                issue(run_dQ, u, j, ik)
                issue(run_release, ik % stages)
                if more and mutate != "mma_dp_before_dq":
                    yield ("full", (ik + 3) % stages), ((ik + 3) // stages) & 1
                    issue(run_dP, u, j + 1, ik + 3)
                    commit("dp_full")
                    issue(run_release, (ik + 3) % stages)
                gblk += 1
            commit("unit_done")
        mma_done[0] = True

    def ew(h):
        gblk = 0
        for u, J in enumerate(units):
            # Q_i, dO_i rows into TMEM: the previous unit's products read them
            # (its unit_done was waited for in the epilogue below).
            if u > 0:
                left = [(k, u - 1, j) for j in range(units[u - 1]) for k in ("S", "dP")
                        if (k, u - 1, j) not in ran]
                if left:
                    raise Violation(f"element-wise {h} replaces Q/dO rows while {left} still read them")
            qdo[h] = u
            bar("fix_full").arrive()
            for j in range(J):
                yield "s_full", gblk & 1
                if s_reg[h] != ("S", u, j):
                    raise Violation(f"element-wise {h} expected S {(u, j)}, TMEM holds {s_reg[h]}")
                s_read[h] = ("S", u, j)
                bar("s_read").arrive()
                yield "dp_full", gblk & 1
                if dp_reg[h] != ("dP", u, j):
                    raise Violation(f"element-wise {h} expected dP {(u, j)}, TMEM holds {dp_reg[h]}")
                dp_reg[h] = ("dS", u, j)        # dS over dP (read)
                bar("p_ready").arrive()
                gblk += 1
            if mutate != "ew_skips_unit_done":
                yield "unit_done", u & 1
            missing = [("dQ", u, j) for j in range(J) if ("dQ", u, j) not in ran]
            if missing:
                raise Violation(f"element-wise {h} reads dQ of unit {u} before {missing}")

    roles = {"load": load(), "mma": mma(), "tensor": tensor()}
    roles.update({f"ew{h}": ew(h) for h in EW})
    return run_roles(roles, bars, seed)


KERNELS = {"dkdv": simulate_dkdv, "dq": simulate_dq}


def random_units(rng):
    return [rng.choice([1, 1, 2, 3, 5, 8]) for _ in range(rng.randint(1, 6))]


# The kernels' ring depths (dK/dV: 5 at d = 128, 12 at d = 64; dQ: 6 and 12) and a
# short ring that makes the producer wait more often.
@pytest.mark.parametrize("kernel,stages", [("dkdv", 5), ("dkdv", 12), ("dkdv", 3), ("dq", 6),
                                           ("dq", 12), ("dq", 3)])
def test_bwd_protocol_completes_and_is_safe(kernel, stages):
    rng = random.Random(2000 + stages + 10 * len(kernel))
    for case in range(150):
        units = random_units(rng)
        stuck = KERNELS[kernel](units, stages, seed=case)
        assert not stuck, (units, stuck)


@pytest.mark.parametrize("mutation,kernel", [
    ("mma_s_before_dv", "dkdv"),
    ("mma_dp_before_dk", "dkdv"),
    ("ew_skips_dp_full", "dkdv"),
    ("load_skips_fix_empty", "dkdv"),
    ("load_skips_empty_wait", "dkdv"),
    ("mma_skips_s_read", "dq"),
    ("mma_dp_before_dq", "dq"),
    ("ew_skips_unit_done", "dq"),
    ("load_skips_empty_wait", "dq"),
])
def test_bwd_protocol_mutations_are_caught(mutation, kernel):
    rng = random.Random(11)
    for case in range(300):
        units = random_units(rng)
        try:
            stuck = KERNELS[kernel](units, 6, mutate=mutation, seed=case)
        except Violation:
            return
        if stuck:
            return
    pytest.fail(f"{mutation} ({kernel}) was not caught")
