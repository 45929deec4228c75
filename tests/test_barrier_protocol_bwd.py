"""A CPU model of the backward kernel's mbarrier protocol, run under random
interleavings: no schedule may deadlock, no parity wait may pass on the wrong
phase, and no buffer may be overwritten while a reader still needs it.

The roles of warp_specialized_attention_gb300/csrc/fmha_bwd_sm103.cuh talk
only through mbarriers (the full/empty channels of "Tawa: Automatic Warp
Specialization for Modern GPUs with Asynchronous References", Section
III-B/III-E), and every wait names its phase by parity alone.  The model
mirrors the kernel's barrier program role by role:

  loader   K and V once; per query block n: Q into buffer n % 2 (q_full/q_free),
           dO into its one buffer (do_full/do_free), LSE and delta into
           statistics buffer n % 2 (plain stores, stat_full/stat_free); then it
           waits for its own copies to land
  MMA      S^T = K Q^T; after do_full and dq_free: dP^T = V dO^T, commit sd_full; after
           p_ready: dV (commit do_free), dK (commit q_free), dQ (commit dq_full,
           ds_free); at the end acc_done and its own drain
  compute  8 warps: statistics, S^T and dP^T in; P^T over S^T and dS^T out;
           p_ready and stat_free; after acc_done the dV/dK epilogue
  dQ       8 warps: dQ out of TMEM, then dq_free
  tensor   MMAs execute, and commits complete, in issue order after random
           delays; TMA copies land in any order

Beyond the barrier rules, the model keeps a tag of what every buffer holds
(Q buffers, dO, statistics, the S^T/P^T and dP^T/dQ TMEM columns, the dS^T
tile).  A writer sets the tag when its write lands; an MMA checks its
operands when it executes, and a CUDA-core role checks at the start and the
end of its read, so an overwrite that lands too early is reported.
"""
import random

import pytest

N_COMPUTE = 8
N_DQ = 8


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


class BwdModel:
    def __init__(self, nq, seed):
        self.rng = random.Random(seed)
        self.nq = nq
        self.errors = []
        self.bars = {}
        self.tensor_q = []     # ("mma", fn) or ("commit", bar), in issue order
        self.tma_q = []        # (bar, land_fn), any order
        b = self.bar
        b("kv_full", 1)
        for i in range(2):
            b(("q_full", i), 1)
            b(("q_free", i), 1)
            b(("stat_full", i), 1)
            b(("stat_free", i), N_COMPUTE)
        for name, count in (("do_full", 1), ("do_free", 1), ("sd_full", 1),
                            ("p_ready", N_COMPUTE), ("ds_free", 1), ("dq_full", 1),
                            ("dq_free", N_DQ), ("acc_done", 1), ("mma_drain", 1)):
            b(name, count)
        # what each buffer holds
        self.res = {"K": None, "V": None, ("Q", 0): None, ("Q", 1): None, "dO": None,
                    ("stat", 0): None, ("stat", 1): None, "dPdQ": None}
        self.s_cols = [None] * N_COMPUTE   # S^T, then P^T, per compute warp's columns
        self.ds_tile = [None] * N_COMPUTE  # dS^T rows/columns written by each warp
        self.dv_steps = 0
        self.dk_steps = 0

    def bar(self, name, count):
        self.bars[name] = Bar(count)

    def wait(self, name, index):
        """Wait for phase `index` of `name` by its parity, as the kernel does."""
        bar = self.bars[name]
        while (bar.done & 1) == (index & 1):
            yield
        if bar.done <= index:
            self.errors.append("wait on %s passed for phase %d with %d phases done"
                               % (name, index, bar.done))

    def expect(self, what, got, want):
        if got != want:
            self.errors.append("%s holds %r, expected %r" % (what, got, want))

    def copy(self, bar, land):
        self.tma_q.append((bar, land))

    def issue(self, fn):
        self.tensor_q.append(("mma", fn))

    def commit(self, bar):
        self.tensor_q.append(("commit", bar))

    # ------------------------------------------------------------------ roles
    def loader(self):
        def put(key, tag):
            def land():
                self.res[key] = tag
            return land
        self.copy("kv_full", lambda: (self.res.__setitem__("K", "kv"),
                                      self.res.__setitem__("V", "kv")))
        for n in range(self.nq):
            qb = n & 1
            if n >= 2:
                yield from self.wait(("q_free", qb), (n >> 1) - 1)
            self.copy(("q_full", qb), put(("Q", qb), ("Q", n)))
            if n >= 1:
                yield from self.wait("do_free", n - 1)
            self.copy("do_full", put("dO", ("dO", n)))
            sb = n & 1
            if n >= 2:
                yield from self.wait(("stat_free", sb), (n >> 1) - 1)
            self.res[("stat", sb)] = ("stat", n)
            yield
            self.bars[("stat_full", sb)].arrive()
        # drain: every issued copy lands before the block may exit
        yield from self.wait("kv_full", 0)
        for b in range(2):
            nb = (self.nq + 1 - b) >> 1
            if nb > 0:
                yield from self.wait(("q_full", b), nb - 1)
        yield from self.wait("do_full", self.nq - 1)

    def mma(self):
        yield from self.wait("kv_full", 0)
        for n in range(self.nq):
            qb = n & 1
            yield from self.wait(("q_full", qb), n >> 1)

            def s_t(n=n, qb=qb):
                self.expect("K", self.res["K"], "kv")
                self.expect("Q buffer %d at S^T" % qb, self.res[("Q", qb)], ("Q", n))
                self.s_cols = [("S", n)] * N_COMPUTE
            self.issue(s_t)
            yield from self.wait("do_full", n)
            yield from self.mma_wait_dq_free(n)

            def dp_t(n=n):
                self.expect("V", self.res["V"], "kv")
                self.expect("dO at dP^T", self.res["dO"], ("dO", n))
                self.res["dPdQ"] = ("dP", n)
            self.issue(dp_t)
            self.commit("sd_full")
            yield from self.wait("p_ready", n)

            def dv(n=n):
                for w in range(N_COMPUTE):
                    self.expect("P^T columns of warp %d" % w, self.s_cols[w], ("P", n))
                self.expect("dO at dV", self.res["dO"], ("dO", n))
                self.dv_steps += 1
            self.issue(dv)
            self.commit("do_free")

            def dk(n=n, qb=qb):
                for w in range(N_COMPUTE):
                    self.expect("dS^T part %d at dK" % w, self.ds_tile[w], ("dS", n))
                self.expect("Q buffer %d at dK" % qb, self.res[("Q", qb)], ("Q", n))
                self.dk_steps += 1
            self.issue(dk)
            self.commit(("q_free", qb))

            def dq(n=n):
                for w in range(N_COMPUTE):
                    self.expect("dS^T part %d at dQ" % w, self.ds_tile[w], ("dS", n))
                self.expect("K at dQ", self.res["K"], "kv")
                self.res["dPdQ"] = ("dQ", n)
            self.issue(dq)
            self.commit("dq_full")
            self.commit("ds_free")
        self.commit("acc_done")
        self.commit("mma_drain")
        yield from self.wait("mma_drain", 0)

    def mma_wait_dq_free(self, n):
        # dP^T takes the columns of the previous block's dQ part
        if n >= 1:
            yield from self.wait("dq_free", n - 1)

    def compute(self, w):
        for n in range(self.nq):
            sb = n & 1
            yield from self.wait(("stat_full", sb), n >> 1)
            yield from self.wait("sd_full", n)
            if n >= 1:
                yield from self.wait("ds_free", n - 1)
            for phase in ("start", "end"):
                self.expect("statistics %d (%s of warp %d's read)" % (sb, phase, w),
                            self.res[("stat", sb)], ("stat", n))
                self.expect("S^T columns of warp %d (%s)" % (w, phase), self.s_cols[w], ("S", n))
                self.expect("dP^T columns (%s of warp %d's read)" % (phase, w),
                            self.res["dPdQ"], ("dP", n))
                if phase == "start":
                    yield
            self.s_cols[w] = ("P", n)
            self.ds_tile[w] = ("dS", n)
            yield
            self.bars["p_ready"].arrive()
            self.bars[("stat_free", sb)].arrive()
        yield from self.wait("acc_done", 0)
        if self.dv_steps != self.nq or self.dk_steps != self.nq:
            self.errors.append("epilogue of warp %d saw %d dV and %d dK steps of %d"
                               % (w, self.dv_steps, self.dk_steps, self.nq))

    def dq_warp(self, w):
        for n in range(self.nq):
            yield from self.wait("dq_full", n)
            self.expect("dQ columns (start of dQ warp %d's read)" % w, self.res["dPdQ"], ("dQ", n))
            yield
            self.expect("dQ columns (end of dQ warp %d's read)" % w, self.res["dPdQ"], ("dQ", n))
            self.bars["dq_free"].arrive()

    def engines(self):
        while True:
            r = self.rng.random()
            if self.tensor_q and r < 0.5:
                kind, x = self.tensor_q.pop(0)
                if kind == "mma":
                    x()
                else:
                    self.bars[x].arrive()
            elif self.tma_q and r >= 0.5:
                bar, land = self.tma_q.pop(self.rng.randrange(len(self.tma_q)))
                land()
                self.bars[bar].arrive()
            yield

    def run(self, max_idle=20000):
        roles = ([self.loader(), self.mma()] + [self.compute(w) for w in range(N_COMPUTE)]
                 + [self.dq_warp(w) for w in range(N_DQ)])
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
                return "error: " + self.errors[0]
            if idle > max_idle and not self.tensor_q and not self.tma_q:
                return "deadlock"
        if self.tensor_q or self.tma_q:
            return "exited with asynchronous work in flight"
        if self.bars["dq_free"].done != self.nq or self.bars["p_ready"].done != self.nq:
            return "incomplete"
        return "ok"


@pytest.mark.parametrize("nq", [1, 2, 3, 4, 5, 7])
def test_backward_protocol_is_safe(nq):
    """nq query blocks per key block: 1 (a causal key block at the diagonal's
    end) up to several, so both Q and statistics buffers wrap around."""
    for seed in range(150):
        res = BwdModel(nq, 1000 * nq + seed).run()
        assert res == "ok", "nq %d seed %d: %s" % (nq, seed, res)


def _first_failure(model_cls, nq, seeds=200):
    for seed in range(seeds):
        res = model_cls(nq, seed).run()
        if res != "ok":
            return res
    return "ok"


def test_model_detects_q_overwritten_before_dk():
    """Negative control: a loader that reuses a Q buffer without waiting for
    q_free must be caught overwriting a Q that dK has not read yet."""
    class NoQFree(BwdModel):
        def wait(self, name, index):
            if isinstance(name, tuple) and name[0] == "q_free":
                return iter(())
            return BwdModel.wait(self, name, index)
    res = _first_failure(NoQFree, 5)
    assert res.startswith("error:") and "Q buffer" in res, res


def test_model_detects_dq_columns_reused_too_early():
    """Negative control: an issuer that writes dP^T without waiting for the
    dQ warps to release the columns must be caught clobbering dQ."""
    class NoDqFree(BwdModel):
        def mma_wait_dq_free(self, n):
            return iter(())
    res = _first_failure(NoDqFree, 4)
    assert res.startswith("error:") and "dQ columns" in res, res


def test_model_detects_a_deadlock():
    """Negative control: a dQ warp that waits for the next block's dQ before
    releasing this one's columns deadlocks the issuer."""
    class Greedy(BwdModel):
        def dq_warp(self, w):
            for n in range(self.nq):
                yield from self.wait("dq_full", n)
                if n + 1 < self.nq:
                    yield from self.wait("dq_full", n + 1)
                self.bars["dq_free"].arrive()
    res = Greedy(3, 0).run(max_idle=3000)
    assert res == "deadlock", res
