"""CPU model of the forward kernel's producer/consumer protocol (no GPU).

"4.3 FlashAttention 2 & 3", section "A from-scratch model of the
producer/consumer pipeline", models FA3's shared-memory ring as a queue: the
producer runs ahead by the number of stages, the consumer takes a tile only
once it is present, and the result is exact attention.  This file models the
same ring the way the kernel drives it -- mbarriers with a phase bit, item i in
slot i mod S with parity (i / S) mod 2, the producer waiting on the slot's
"empty" barrier with the opposite parity, the consumer on its "full" barrier,
asynchronous completions (the copy engine fills a slot later; the tensor pipe
frees it later) -- with threads and random delays, and checks:
  * every tile is consumed once, in order, with the payload the producer wrote;
  * the producer never overwrites a slot whose tile has not been released;
  * the final drain (the producer waiting for its own last copies before the
    block exits) computes the right (slot, parity) and never blocks;
  * the consumer's streamed (m, l, O) state over the tiles equals the oracle's
    three-pass attention (the oracle's block state and merge rule);
  * the work-unit hand-off ring (4 entries, one producer, nine consumers) gives
    every consumer the same units, and its end marker.
Mutations of the parity arithmetic must be caught (deadlock, detected by the
bounded waits, or a stale read).
"""
import random
import threading
import time

import numpy as np
import pytest

from oracle import attention as oa


class MBarrier:
    """An mbarrier: `count` arrivals complete the current phase; a wait with
    parity P succeeds once the phase of parity P has completed, i.e. while the
    current phase's parity differs from P (so a fresh barrier, phase 0, lets a
    wait with parity 1 through at once)."""

    def __init__(self, count: int):
        self.count = count
        self.pending = count
        self.phase = 0
        self.lock = threading.Lock()

    def arrive(self):
        with self.lock:
            self.pending -= 1
            assert self.pending >= 0
            if self.pending == 0:
                self.phase += 1
                self.pending = self.count

    def try_wait(self, parity: int) -> bool:
        with self.lock:
            return (self.phase & 1) != parity


def wait_bounded(bar: MBarrier, parity: int, limit_s: float = 2.0) -> bool:
    """The kernel's bounded wait: spin, give up after a time limit."""
    t0 = time.monotonic()
    while not bar.try_wait(parity):
        if time.monotonic() - t0 > limit_s:
            return False
        time.sleep(0)
    return True


class Async:
    """A completion engine (copy engine / tensor pipe): runs callbacks in
    order, each after a random delay."""

    def __init__(self, rng):
        self.q = []
        self.cv = threading.Condition()
        self.rng = rng
        self.stop = False
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()

    def post(self, fn):
        with self.cv:
            self.q.append(fn)
            self.cv.notify()

    def _run(self):
        while True:
            with self.cv:
                while not self.q and not self.stop:
                    self.cv.wait(0.01)
                if not self.q and self.stop:
                    return
                fn = self.q.pop(0)
            time.sleep(self.rng.random() * 2e-4)
            fn()

    def close(self):
        with self.cv:
            self.stop = True
            self.cv.notify()
        self.t.join(5)


def run_ring(tiles, stages, seed, producer_parity=lambda ph: ph ^ 1,
             consumer_parity=lambda ph: ph):
    """Producer and consumer threads over a ring of `stages` slots carrying
    `tiles` (a list of payloads).  Returns (consumed payloads, error list)."""
    rng = random.Random(seed)
    full = [MBarrier(1) for _ in range(stages)]
    empty = [MBarrier(1) for _ in range(stages)]
    slots = [None] * stages
    released = set()            # items whose slot the consumer has handed back
    errors, consumed = [], []
    copy_engine, tensor_pipe = Async(random.Random(seed + 1)), Async(random.Random(seed + 2))
    n = len(tiles)

    def producer():
        for item in range(n):
            slot, ph = item % stages, (item // stages) & 1
            if not wait_bounded(empty[slot], producer_parity(ph)):
                errors.append(f"producer timed out at item {item}")
                return
            if item >= stages and (item - stages) not in released:
                errors.append(f"slot {slot} overwritten before item {item - stages} was released")
            time.sleep(rng.random() * 1e-4)

            def land(slot=slot, item=item):
                slots[slot] = (item, tiles[item])
                full[slot].arrive()          # the copy's bytes complete the phase
            copy_engine.post(land)
        # Drain: wait for the last copy into every slot that was used.
        for s in range(min(stages, n)):
            last = s + ((n - 1 - s) // stages) * stages
            if not wait_bounded(full[s], (last // stages) & 1):
                errors.append(f"drain of slot {s} timed out")

    def consumer():
        for item in range(n):
            slot, ph = item % stages, (item // stages) & 1
            if not wait_bounded(full[slot], consumer_parity(ph)):
                errors.append(f"consumer timed out at item {item}")
                return
            got = slots[slot]
            if got is None or got[0] != item:
                errors.append(f"item {item}: slot {slot} holds {None if got is None else got[0]}")
                return
            consumed.append(got[1])
            time.sleep(rng.random() * 1e-4)

            def free(slot=slot, item=item):
                released.add(item)
                empty[slot].arrive()         # the commit after the products that read it
            tensor_pipe.post(free)

    tp, tc = threading.Thread(target=producer), threading.Thread(target=consumer)
    tp.start(), tc.start()
    tp.join(30), tc.join(30)
    copy_engine.close(), tensor_pipe.close()
    return consumed, errors


@pytest.mark.parametrize("stages", [2, 4, 8])
@pytest.mark.parametrize("seed", [0, 1])
def test_ring_streams_exact_attention(stages, seed):
    """Key/value tiles through the ring; the consumer folds each tile into its
    (m, l, O) state with the oracle's block state and merge rule; the result is
    the oracle's three-pass attention."""
    rng = np.random.default_rng(seed)
    N, d, Bc = 200, 8, 16
    q = rng.standard_normal((5, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    scale = d ** -0.5
    tiles = [(k[j:j + Bc], v[j:j + Bc]) for j in range(0, N, Bc)]
    consumed, errors = run_ring(tiles, stages, seed)
    assert not errors, errors
    assert len(consumed) == len(tiles)
    for i in range(q.shape[0]):
        state = (-np.inf, 0.0, np.zeros(d))
        for kj, vj in consumed:
            state = oa.merge(state, oa.partial_state(scale * (kj @ q[i]), vj))
        m, ell, o = state
        O_ref, L_ref = oa.three_pass_rows(q, k, v, scale, False, [i])
        np.testing.assert_allclose(o / ell, O_ref[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(m + np.log(ell), L_ref[0], rtol=1e-12)


@pytest.mark.parametrize("stages", [4, 8])
def test_ring_many_items(stages):
    tiles = list(range(200))
    consumed, errors = run_ring(tiles, stages, seed=stages)
    assert not errors, errors
    assert consumed == tiles


def test_producer_waiting_on_the_wrong_parity_is_caught():
    """With the consumer's parity the producer's first wait, on a fresh empty
    barrier, never completes: the bounded wait reports it."""
    _, errors = run_ring(list(range(12)), 4, seed=3, producer_parity=lambda ph: ph)
    assert any("producer timed out" in e for e in errors)


def test_consumer_waiting_on_the_wrong_parity_is_caught():
    """With the producer's parity the consumer passes a fresh full barrier at
    once and reads a slot before its copy has landed."""
    _, errors = run_ring(list(range(12)), 4, seed=4, consumer_parity=lambda ph: ph ^ 1)
    assert any("holds" in e or "timed out" in e for e in errors)


def test_drain_parity_formula():
    """The drain waits on slot s for the parity of its last fill, item
    s + floor((n - 1 - s) / S) * S -- checked against a direct count."""
    for S in (2, 4, 8):
        for n in range(1, 40):
            for s in range(min(S, n)):
                last = s + ((n - 1 - s) // S) * S
                fills = [i for i in range(n) if i % S == s]
                assert last == fills[-1]
                assert (last // S) & 1 == (len(fills) - 1) & 1


def test_unit_handoff_ring():
    """Work units: the load warp publishes each unit index (then -1) in a
    4-entry ring; nine consumers (the MMA warp and eight softmax warps) read
    every entry and each frees it; the producer reuses an entry only after all
    nine have freed it."""
    units = list(range(37))
    consumers = 9
    full = [MBarrier(1) for _ in range(4)]
    empty = [MBarrier(consumers) for _ in range(4)]
    ring = [None] * 4
    seen = [[] for _ in range(consumers)]
    errors = []
    reads = {}                    # k -> how many consumers have read entry k
    lock = threading.Lock()
    rng = random.Random(7)

    def producer():
        seq = units + [-1]
        for k, u in enumerate(seq):
            slot = k & 3
            if k >= 4:
                if not wait_bounded(empty[slot], ((k >> 2) - 1) & 1):
                    errors.append(f"producer timed out at {k}")
                    return
                with lock:
                    if reads.get(k - 4, 0) != consumers:
                        errors.append(f"entry {k - 4} reused before all consumers read it")
            ring[slot] = u
            full[slot].arrive()

    def consumer(c):
        k = 0
        while True:
            slot = k & 3
            if not wait_bounded(full[slot], (k >> 2) & 1):
                errors.append(f"consumer {c} timed out at {k}")
                return
            u = ring[slot]
            with lock:
                reads[k] = reads.get(k, 0) + 1
            seen[c].append(u)
            time.sleep(rng.random() * 1e-4)
            empty[slot].arrive()
            if u < 0:
                return
            k += 1

    ts = [threading.Thread(target=producer)] + [threading.Thread(target=consumer, args=(c,))
                                                for c in range(consumers)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(30)
    assert not errors, errors
    for c in range(consumers):
        assert seen[c] == units + [-1]
