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
             (kv_full, and one kv_empty per query tile: a slot is reloaded
             once every tile that read its previous item has released it),
             Q_t after K_0/V_0 of each unit (q_full[t]/q_empty[t])
  MMA        the head-dim 128 schedule (P over S): one issuer for both tiles
             in the order P_0 V(j), S_0(j+1), P_1 V(j), S_1(j+1), releasing
             every ring item and both Q tiles; the head-dim 64 one (split P:
             s_free, P handed over whole, pvb_done): one issuer per query
             tile, each releasing the ring items and the Q tile its tile read
  softmax    4 warps per query tile: S wait, P releases (in two halves over
             S, whole with split P), the rescale waits, epilogue
             (o_full/o_empty); in a key-split unit
             (both tiles on the same 128 query rows, tile 0 on the first half
             of the keys, tile 1 on the second) tile 1 hands its row
             statistics over (merge) and tile 0 writes the merged result and
             frees both O tiles
  tensor     each issuer's commits complete in its own issue order after
             random delays; two issuers' commits interleave freely
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
        self.units = [u if len(u) == 3 else (u[0], u[1], False) for u in units]
        # (nkv0, nkv1, key_split): a key-split unit has nkv0 == nkv1 blocks per tile
        self.split = split
        self.stages = stages
        self.merge_every_unit = not split and not causal   # the kernels that may key-split
        self.errors = []
        self.bars = {}
        self.tma_q = []              # pending copies, completed in any order
        self.tensor_q = [[], []]     # per issuer: pending commits, completed in order
        b = self.bar
        for i in range(2):
            b(("unit_full", i), 1)
            b(("unit_empty", i), 10 if split else 9)   # issuers + eight softmax warps
        b(("merge",), 4)                                 # tile 1's warps, key-split units
        for t in range(2):
            for n, c in (("s_full", 1), ("p0", 4), ("p1", 4), ("pva", 1), ("pvb", 1),
                         ("s_free", 4), ("o_full", 1), ("o_empty", 4), ("q_full", 1),
                         ("q_empty", 1)):
                b((n, t), c)
        for s in range(stages):
            b(("kv_full", s), 1)
            for t in range(2):
                b(("kv_empty", t, s), 1)
        self.unit_slot = [None, None]
        self.slot_item = [None] * stages   # which ring item each slot holds (set when a copy lands)
        self.stats = [None] * 4            # per warp quadrant: whose row statistics tile 1 left

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

    def commit(self, t, name):
        self.tensor_q[t].append(name)

    def copy(self, name, item=None):
        self.tma_q.append((name, item))

    def check_slot(self, t, item, what):
        """The ring slot of `item` must still hold it when tile t's MMAs read or release it."""
        slot = item % self.stages
        if self.slot_item[slot] != item:
            self.errors.append("tile %d %s item %d but slot %d holds item %s"
                               % (t, what, item, slot, self.slot_item[slot]))

    # ------------------------------------------------------------------ roles
    def producer(self):
        it = 0
        nq = [0, 0]
        mask = [0] * self.stages          # tiles that read the item now in each slot
        uses = [[0] * self.stages for _ in range(2)]   # items of each slot each tile read
        for k in range(len(self.units) + 1):
            if k >= 2:   # the consumers have read the unit that used this slot before
                yield from self.wait(("unit_empty", k & 1), (k >> 1) - 1)
            self.unit_slot[k & 1] = k if k < len(self.units) else -1
            self.bars[("unit_full", k & 1)].arrive()
            if k == len(self.units):
                return
            n0, n1, ks = self.units[k]
            for j in range(n1):
                # a key-split unit loads K_j, K_{h+j}, V_j, V_{h+j} per step
                for kv in range(4 if ks else 2):
                    slot = it % self.stages
                    for t in range(2):
                        if mask[slot] >> t & 1:
                            yield from self.wait(("kv_empty", t, slot), uses[t][slot] - 1)
                    # one issuer releases every item (as issuer 0); two
                    # issuers release the items their own tile read
                    mask[slot] = (2 | (1 if j < n0 else 0)) if self.split else 1
                    for t in range(2):
                        uses[t][slot] += mask[slot] >> t & 1
                    self.copy(("kv_full", slot), it)
                    it += 1
                    if j == 0 and kv == (3 if ks else 1):
                        for t in range(2):
                            if nq[t] > 0:
                                yield from self.wait(("q_empty", t), nq[t] - 1)
                            self.copy(("q_full", t))
                            nq[t] += 1

    def next_unit(self, k):
        yield from self.wait(("unit_full", k & 1), k >> 1)
        u = self.unit_slot[k & 1]
        self.bars[("unit_empty", k & 1)].arrive()
        return u

    def mma_tile(self, t):
        """The issuer of query tile t (split P)."""
        it = g = 0
        k = 0
        while True:
            u = yield from self.next_unit(k)
            if u < 0:
                return
            n = self.units[u][t]
            n1 = self.units[u][1]
            K = lambda j: it + 2 * j
            V = lambda j: it + 2 * j + 1
            full = lambda item: self.wait(("kv_full", item % self.stages), item // self.stages)
            release = lambda item: self.commit(t, ("release", t, item))

            def use(item):
                yield from full(item)
                self.check_slot(t, item, "reads")
            yield from use(K(0))
            yield from self.wait(("q_full", t), k)
            if self.split and g > 0:
                yield from self.wait(("s_free", t), g - 1)
            self.commit(t, ("s_full", t))
            release(K(0))
            if n == 1:
                self.commit(t, ("q_empty", t))
            if k > 0:
                yield from self.wait(("o_empty", t), k - 1)
            for j in range(n):
                if self.split and j + 1 < n:
                    yield from use(K(j + 1))
                    yield from self.wait(("s_free", t), g + j)
                    self.commit(t, ("s_full", t))
                    release(K(j + 1))
                    if j + 2 == n:
                        self.commit(t, ("q_empty", t))
                yield from use(V(j))
                if self.split:                            # P handed over whole
                    yield from self.wait(("p1", t), g + j)
                    self.commit(t, ("pvb", t))
                else:
                    yield from self.wait(("p0", t), g + j)
                    self.commit(t, ("pva", t))
                    yield from self.wait(("p1", t), g + j)
                release(V(j))
                if j == n - 1:
                    self.commit(t, ("o_full", t))
                if not self.split and j + 1 < n:
                    yield from use(K(j + 1))
                    self.commit(t, ("s_full", t))
                    release(K(j + 1))
                    if j + 2 == n:
                        self.commit(t, ("q_empty", t))
            it += 2 * n1
            g += n
            k += 1

    def mma_single(self):
        """One issuer for both tiles (P over S)."""
        it = g0 = g1 = 0
        k = 0
        while True:
            u = yield from self.next_unit(k)
            if u < 0:
                return
            n0, n1, ks = self.units[u]
            # ring items: both tiles read K_j, V_j; a key-split unit gives each
            # tile its own K and V per step (tile 1 on keys h + j)
            K = lambda t, j: it + 4 * j + t if ks else it + 2 * j
            V = lambda t, j: it + 4 * j + 2 + t if ks else it + 2 * j + 1
            full = lambda item: self.wait(("kv_full", item % self.stages), item // self.stages)
            release = lambda item: self.commit(0, ("release", 0, item))

            def use(item):
                yield from full(item)
                self.check_slot(0, item, "reads")

            def pv(t, g, j):
                yield from self.wait(("p0", t), g + j)
                self.commit(0, ("pva", t))
                yield from self.wait(("p1", t), g + j)

            def free_q():
                self.commit(0, ("q_empty", 0))
                self.commit(0, ("q_empty", 1))

            yield from use(K(0, 0))
            if ks:
                yield from use(K(1, 0))
            yield from self.wait(("q_full", 0), k)
            yield from self.wait(("q_full", 1), k)
            self.commit(0, ("s_full", 0))
            self.commit(0, ("s_full", 1))
            release(K(0, 0))
            if ks:
                release(K(1, 0))
            if n1 == 1:
                free_q()
            if k > 0:
                yield from self.wait(("o_empty", 0), k - 1)
                yield from self.wait(("o_empty", 1), k - 1)
            for j in range(n1):
                more = j + 1 < n1
                yield from use(V(0, j))
                if j < n0:
                    yield from pv(0, g0, j)
                    if j == n0 - 1:
                        self.commit(0, ("o_full", 0))
                if ks:
                    release(V(0, j))
                if more:
                    yield from use(K(0, j + 1))
                    if j + 1 < n0:
                        self.commit(0, ("s_full", 0))
                    if ks:
                        release(K(0, j + 1))
                if ks:
                    yield from use(V(1, j))
                yield from pv(1, g1, j)
                release(V(1, j))
                if j == n1 - 1:
                    self.commit(0, ("o_full", 1))
                if more:
                    if ks:
                        yield from use(K(1, j + 1))
                    self.commit(0, ("s_full", 1))
                    release(K(1, j + 1))
                    if j + 2 == n1:
                        free_q()
            it += 2 * (n0 + n1) if ks else 2 * n1
            g0 += n0
            g1 += n1
            k += 1

    def softmax(self, t, q):
        """Softmax warp q (TMEM lane quadrant q) of query tile t."""
        g = 0
        k = 0
        rng = self.rng
        while True:
            u = yield from self.next_unit(k)
            if u < 0:
                return
            nkv = self.units[u][t]
            ks = self.units[u][2]
            for j in range(nkv):
                gj = g + j
                yield from self.wait(("s_full", t), gj)
                if self.split:
                    self.bars[("s_free", t)].arrive()
                    # the previous block's whole P V has read the P columns
                    # before any P is rewritten; a raised maximum rescales
                    # O_t, which holds exactly the earlier blocks then
                    if gj > 0:
                        yield from self.wait(("pvb", t), gj - 1)
                    for _ in range(rng.randint(0, 2)):
                        yield
                    self.bars[("p1", t)].arrive()        # all of P at once
                    continue
                self.bars[("p0", t)].arrive()
                for _ in range(rng.randint(0, 2)):
                    yield
                if j > 0 and rng.random() < 0.2:          # keys 64-127 raise the maximum
                    yield from self.wait(("pva", t), gj)
                self.bars[("p1", t)].arrive()
            g += nkv
            yield from self.wait(("o_full", t), k)
            if t == 1 and self.merge_every_unit:
                # tile 1 arrives in every unit: phase k of the barrier is unit k's
                if ks:
                    self.stats[q] = u                # row statistics handed to tile 0
                self.bars[("merge",)].arrive()
            if not ks:
                self.bars[("o_empty", t)].arrive()
            elif t == 0:
                yield from self.wait(("o_full", 1), k)
                yield from self.wait(("merge",), k)
                if self.stats[q] != u:
                    self.errors.append("tile 0 merged unit %d with statistics of unit %s"
                                       % (u, self.stats[q]))
                self.bars[("o_empty", 0)].arrive()   # both O tiles read: free them
                self.bars[("o_empty", 1)].arrive()
            k += 1

    def engines(self):
        """The tensor pipe completes commits in issue order; TMA copies land
        in any order."""
        while True:
            r = self.rng.random()
            queues = [q for q in self.tensor_q if q]
            if queues and r < 0.5:
                name = self.rng.choice(queues).pop(0)
                if name[0] == "release":   # tile t's MMAs reading this item have completed
                    _, t, item = name
                    self.check_slot(t, item, "released")
                    self.bars[("kv_empty", t, item % self.stages)].arrive()
                else:
                    self.bars[name].arrive()
            elif self.tma_q and r >= 0.5:
                name, item = self.tma_q.pop(self.rng.randrange(len(self.tma_q)))
                if name[0] == "kv_full":
                    self.slot_item[name[1]] = item
                self.bars[name].arrive()
            yield

    def run(self, max_idle=20000):
        issuers = [self.mma_tile(0), self.mma_tile(1)] if self.split else [self.mma_single()]
        roles = [self.producer()] + issuers + [self.softmax(t, q) for t in range(2) for q in range(4)]
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
            if idle > max_idle and not any(self.tensor_q) and not self.tma_q:
                return "deadlock"
        n = len(self.units)
        for t in range(2):
            if self.bars[("o_full", t)].done != n or self.bars[("o_empty", t)].done != n:
                return "incomplete: tile %d finished %d of %d units" % (
                    t, self.bars[("o_empty", t)].done, n)
        return "ok"


def _units(rng, causal, n_units, key_split=False):
    """Random units; with key_split, the tail units (after a random number of
    whole ones, as the host places them) split the keys between the tiles."""
    out = []
    n_whole = rng.randint(0, n_units) if key_split else n_units
    for i in range(n_units):
        qb = rng.randint(0, 4)
        if i >= n_whole:
            out.append((qb + 1, qb + 1, True))
        else:
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


def test_protocol_with_key_split_tail_units():
    """Full attention, head dim 128: whole units followed by key-split ones
    (each tile on half of the keys of the same 128 query rows, merged in the
    block)."""
    for seed in range(400):
        rng = random.Random(seed)
        units = _units(rng, False, rng.randint(1, 6), key_split=True)
        res = Model(units, False, 4, seed, False).run()
        assert res == "ok", "seed %d units %s: %s" % (seed, units, res)


def test_model_detects_a_merge_without_the_other_tile():
    """Negative control: a tile 0 that frees O_1 without waiting for tile 1's
    last P V lets the next unit's P V overwrite O_1 while it may still be
    read; the model must report the false pass or a deadlock."""
    class NoWait(Model):
        def wait(self, name, index):
            if name == ("merge",):
                return iter(())            # the dropped wait
            return Model.wait(self, name, index)
    bad = 0
    for seed in range(200):
        rng = random.Random(seed)
        units = [(2, 2, True)] * rng.randint(2, 4)
        if NoWait(units, False, 4, seed, False).run() != "ok":
            bad += 1
    assert bad > 0


def test_model_detects_a_deadlock():
    """Negative control: a softmax that waits for the P V of the keys it has
    not released yet (its own second half) must be reported as a deadlock."""
    class SelfWait(Model):
        def softmax(self, t, q):
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


def test_model_detects_a_slot_reloaded_before_a_tile_released_it():
    """Negative control: a producer that waits only for tile 1's release of a
    ring slot reloads it while tile 0's MMAs may still read the old item."""
    class OneTileEmpty(Model):
        def wait(self, name, index):
            if name[0] == "kv_empty" and name[1] == 0:
                return iter(())            # the dropped wait
            return Model.wait(self, name, index)
    bad = 0
    for seed in range(200):
        rng = random.Random(seed)
        units = _units(rng, True, rng.randint(2, 5))
        if OneTileEmpty(units, True, 8, seed, True).run() != "ok":
            bad += 1
    assert bad > 0
