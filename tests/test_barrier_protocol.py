"""A CPU model of the attention kernel's mbarrier protocol, run under random
interleavings: no schedule may deadlock, and no wait may pass before the
phase it waits for has completed.

The kernel's roles talk only through mbarriers, and every wait names a
phase by its parity alone (the asynchronous-reference channel of "Tawa:
Automatic Warp Specialization for Modern GPUs with Asynchronous References",
Section III-B/III-E: put / get / consumed lowered to full and empty barriers
with alternating parity).  A parity wait is only correct while its barrier is
at most one phase ahead of the waiter, and a wrong issue order deadlocks only
on data-dependent paths (an O rescale in the middle of a block) or at unit
boundaries of the persistent loop.  Neither shows reliably on a GPU run; both
show here.

The model mirrors, role by role, the barrier program of
warp_specialized_attention_gb300/csrc/fmha_fwd_sm103.cuh:

  producer   unit channel (unit_full/unit_empty), K_j/V_j through a ring
             (kv_full/kv_empty), Q after K_0/V_0 of each unit (q_full/q_empty)
  MMA        Q K^T and P V issue with tcgen05.commit arrivals; the head-dim 128
             schedule (P over S) and the head-dim 64 one (split P: s_free,
             pva_done/pvb_done)
  softmax    4 warps per query tile: S wait, P releases in two halves, the
             rescale waits, epilogue (o_full/o_empty)
  tensor     commits complete in issue order after random delays
  TMA        copies complete in any order after random delays

Barrier semantics are the hardware's: a wait for parity p passes iff the
number of completed phases has parity != p.  The model records, for every
passed wait, which phase the code meant; a pass before that phase completed
is reported.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.done = 0          # completed phases

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


class Model:
    def __init__(self, units, split, stages, seed, causal):
        self.rng = random.Random(seed)
        self.units = units           # list of (nkv0, nkv1)
        self.split = split
        self.stages = stages
        self.errors = []
        self.bars = {}
        self.tensor_q = []           # pending commits, completed in order
        self.tma_q = []              # pending copies, completed in any order
        b = self.bar
        for i in range(2):
            b(("unit_full", i), 1)
            b(("unit_empty", i), 9)
        b("q_full", 1)
        b("q_empty", 1)
        for t in range(2):
            for n, c in (("s_full", 1), ("p0", 4), ("p1", 4), ("pva", 1), ("pvb", 1),
                         ("s_free", 4), ("o_full", 1), ("o_empty", 4)):
                b((n, t), c)
        for s in range(stages):
            b(("kv_full", s), 1)
            b(("kv_empty", s), 1)
        self.unit_slot = [None, None]

    def bar(self, name, count):
        self.bars[name] = Bar(count)

    def wait(self, name, index):
        """Wait for phase `index` of barrier `name` (by its parity, as the kernel does)."""
        bar = self.bars[name]
        while (bar.done & 1) == (index & 1):
            yield
        if bar.done <= index:
            self.errors.append("wait on %s passed for phase %d with %d phases done"
                               % (name, index, bar.done))

    def commit(self, name):
        self.tensor_q.append(name)

    def copy(self, name):
        self.tma_q.append(name)

    # ------------------------------------------------------------------ roles
    def producer(self):
        it = nq = 0
        for k in range(len(self.units) + 1):
            if k >= 2:   # the consumers have read the unit that used this slot before
                yield from self.wait(("unit_empty", k & 1), (k >> 1) - 1)
            self.unit_slot[k & 1] = k if k < len(self.units) else -1
            self.bars[("unit_full", k & 1)].arrive()
            if k == len(self.units):
                return
            n1 = self.units[k][1]
            for j in range(n1):
                for kv in range(2):
                    slot, use = it % self.stages, it // self.stages
                    if use > 0:
                        yield from self.wait(("kv_empty", slot), use - 1)
                    self.copy(("kv_full", slot))
                    it += 1
                    if j == 0 and kv == 1:
                        if nq > 0:
                            yield from self.wait("q_empty", nq - 1)
                        self.copy("q_full")
                        nq += 1

    def next_unit(self, k):
        yield from self.wait(("unit_full", k & 1), k >> 1)
        u = self.unit_slot[k & 1]
        self.bars[("unit_empty", k & 1)].arrive()
        return u

    def mma(self):
        it = g0 = g1 = 0
        k = 0
        while True:
            u = yield from self.next_unit(k)
            if u < 0:
                return
            n0, n1 = self.units[u]
            K = lambda j: it + 2 * j
            V = lambda j: it + 2 * j + 1
            full = lambda item: self.wait(("kv_full", item % self.stages), item // self.stages)
            yield from full(K(0))
            yield from self.wait("q_full", k)

            def pv(t, g, j):
                yield from self.wait(("p0", t), g + j)
                self.commit(("pva", t))
                yield from self.wait(("p1", t), g + j)
                if self.split:
                    self.commit(("pvb", t))

            if self.split:
                if g0 > 0:
                    yield from self.wait(("s_free", 0), g0 - 1)
                self.commit(("s_full", 0))
                if g1 > 0:
                    yield from self.wait(("s_free", 1), g1 - 1)
                self.commit(("s_full", 1))
            else:
                self.commit(("s_full", 0))
                self.commit(("s_full", 1))
            self.commit(("kv_empty", K(0) % self.stages))
            if n1 == 1:
                self.commit("q_empty")
            if k > 0:
                yield from self.wait(("o_empty", 0), k - 1)
                yield from self.wait(("o_empty", 1), k - 1)
            for j in range(n1):
                more = j + 1 < n1
                if self.split:
                    if j + 1 < n0:
                        yield from full(K(j + 1))
                        yield from self.wait(("s_free", 0), g0 + j)
                        self.commit(("s_full", 0))
                    yield from full(V(j))
                    if j < n0:
                        yield from pv(0, g0, j)
                        if j == n0 - 1:
                            self.commit(("o_full", 0))
                    if more:
                        yield from full(K(j + 1))
                        yield from self.wait(("s_free", 1), g1 + j)
                        self.commit(("s_full", 1))
                        self.commit(("kv_empty", K(j + 1) % self.stages))
                        if j + 2 == n1:
                            self.commit("q_empty")
                    yield from pv(1, g1, j)
                    self.commit(("kv_empty", V(j) % self.stages))
                    if j == n1 - 1:
                        self.commit(("o_full", 1))
                else:
                    yield from full(V(j))
                    if j < n0:
                        yield from pv(0, g0, j)
                        if j == n0 - 1:
                            self.commit(("o_full", 0))
                    if more:
                        yield from full(K(j + 1))
                        if j + 1 < n0:
                            self.commit(("s_full", 0))
                    yield from pv(1, g1, j)
                    self.commit(("kv_empty", V(j) % self.stages))
                    if j == n1 - 1:
                        self.commit(("o_full", 1))
                    if more:
                        self.commit(("s_full", 1))
                        self.commit(("kv_empty", K(j + 1) % self.stages))
                        if j + 2 == n1:
                            self.commit("q_empty")
            it += 2 * n1
            g0 += n0
            g1 += n1
            k += 1

    def softmax(self, t):
        g = 0
        k = 0
        rng = self.rng
        while True:
            u = yield from self.next_unit(k)
            if u < 0:
                return
            nkv = self.units[u][t]
            for j in range(nkv):
                gj = g + j
                yield from self.wait(("s_full", t), gj)
                if self.split:
                    self.bars[("s_free", t)].arrive()
                    if gj > 0:
                        yield from self.wait(("pva", t), gj - 1)
                    if j > 0 and rng.random() < 0.2:      # keys 0-63 raise the maximum
                        yield from self.wait(("pvb", t), gj - 1)
                    self.bars[("p0", t)].arrive()
                    if gj > 0:
                        yield from self.wait(("pvb", t), gj - 1)
                else:
                    self.bars[("p0", t)].arrive()
                for _ in range(rng.randint(0, 2)):
                    yield
                if j > 0 and rng.random() < 0.2:          # keys 64-127 raise the maximum
                    yield from self.wait(("pva", t), gj)
                self.bars[("p1", t)].arrive()
            g += nkv
            yield from self.wait(("o_full", t), k)
            self.bars[("o_empty", t)].arrive()
            k += 1

    def engines(self):
        """The tensor pipe completes commits in issue order; TMA copies land
        in any order."""
        while True:
            r = self.rng.random()
            if self.tensor_q and r < 0.5:
                self.bars[self.tensor_q.pop(0)].arrive()
            elif self.tma_q and r >= 0.5:
                self.bars[self.tma_q.pop(self.rng.randrange(len(self.tma_q)))].arrive()
            yield

    def run(self, max_idle=20000):
        roles = [self.producer(), self.mma()] + [self.softmax(t) for t in range(2) for _ in range(4)]
        engines = self.engines()
        alive = list(roles)
        idle = 0
        while alive:
            next(engines)
            p = self.rng.choice(alive)
            try:
                next(p)
                idle += 1
            except StopIteration:
                alive.remove(p)
                idle = 0
            if self.errors:
                return "false pass: " + self.errors[0]
            if idle > max_idle and not self.tensor_q and not self.tma_q:
                return "deadlock"
        n = len(self.units)
        for t in range(2):
            if self.bars[("o_full", t)].done != n or self.bars[("o_empty", t)].done != n:
                return "incomplete: tile %d finished %d of %d units" % (
                    t, self.bars[("o_empty", t)].done, n)
        return "ok"


def _units(rng, causal, n_units):
    out = []
    for _ in range(n_units):
        qb = rng.randint(0, 4)
        out.append((2 * qb + 1, 2 * qb + 2) if causal else (qb + 1, qb + 1))
    return out


@pytest.mark.parametrize("split", [False, True], ids=["D128-P-over-S", "D64-split-P"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_protocol_has_no_deadlock_and_no_false_pass(split, causal):
    stages = 8 if split else 4
    for seed in range(300):
        rng = random.Random(seed)
        units = _units(rng, causal, rng.randint(1, 5))
        res = Model(units, split, stages, seed, causal).run()
        assert res == "ok", "seed %d units %s: %s" % (seed, units, res)


def test_model_detects_a_deadlock():
    """Negative control: a softmax that waits for the P V of the keys it has
    not released yet (its own second half) must be reported as a deadlock."""
    class SelfWait(Model):
        def softmax(self, t):
            u = yield from self.next_unit(0)
            yield from self.wait(("s_full", t), 0)
            self.bars[("p0", t)].arrive()
            yield from self.wait(("pvb", t), 0)        # never committed before p1
            self.bars[("p1", t)].arrive()
    res = SelfWait([(1, 1)], True, 8, 0, False).run(max_idle=2000)
    assert res == "deadlock"


def test_model_detects_a_false_parity_pass():
    """Negative control: a waiter two phases behind its barrier passes on the
    wrong phase, and the model must say so."""
    m = Model([(1, 1)], False, 4, 0, False)
    m.bars[("o_full", 0)].arrive()       # phase 0 done, phase 1 in progress
    # a wait for phase 2 uses parity 0; one completed phase has parity 1, so
    # the hardware rule lets it through although phase 2 has not even begun
    with pytest.raises(StopIteration):
        next(m.wait(("o_full", 0), 2))
    assert m.errors and "phase 2" in m.errors[0]
