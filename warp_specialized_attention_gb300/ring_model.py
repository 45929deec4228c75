"""CPU performance model of a warp-specialized producer/consumer pipeline
through a ring of shared-memory slots, and its use for the attention kernel's
K/V ring.

Source: "A Performance Model for Warp Specialization Kernels", sections
"core formulas" and "three coupled recurrences".  A DMA warp loads an A tile
and then a B tile per stage into a circular buffer of capacity M stages.  A
MATH warp consumes one stage at a time.  The start times obey

    S_a(i) = 0                                               i = 1
           = max(S_b(i-1) + T_LB, S_m(i-M) + T_MATH)          otherwise   (1)
    S_b(i) = max(S_a(i) + T_LA,   S_m(i-M) + T_MATH)                      (2)
    S_m(i) = max(S_m(i-1) + T_MATH, S_b(i) + T_LB)                        (3)

(a load waits for the previous load and for the slot that the stage M back
releases when its MATH ends; MATH waits for its own data and for the previous
MATH).  With W waves of tiles over the SMs, T = (S_m(S) + T_EPI) * W + T_INIT,
where S is the stage count (the last MATH ends at S_m(S) + T_MATH; the page's
T_EPI term absorbs that and the epilogue).  Each time is linear in the tile
size: a throughput plus a startup latency, from two measurements (the page's
two-point calibration).

For attention this module reads the recurrence as follows:
  * A stage is one key block j.  Its "A" and "B" tiles are K_j and V_j.
  * A K/V ring of R slots holds R/2 stages (K and V take one slot each).
  * MATH is the block period of the whole consumer side (both query tiles'
    Q K^T, softmax and P V).  Both slots are taken to return when the
    stage's MATH ends, as in (1)-(2); the kernel frees K_j earlier (after the
    second Q K^T), so the model is pessimistic at small rings.
  * A persistent block runs its units back to back: the next unit's loads
    start as soon as ring slots free up, so one SM's total is one recurrence
    over all its stages.  The page's per-wave T_INIT and T_EPI are paid once
    per block (a launch, a TMEM allocation, a last epilogue).
Nothing here runs on the GPU; it plans, and explains measured ring depths.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

NEG_INF = float("-inf")


def ws_recurrence(n_stages: int, capacity: int, t_la: float, t_lb: float,
                  t_math: float) -> tuple[list[float], list[float], list[float]]:
    """Start times S_a, S_b, S_m (index 0 = stage 1) of equations (1)-(3).

    `capacity` is M, the number of stages the ring holds (>= 1)."""
    if n_stages < 0 or capacity < 1:
        raise ValueError("need n_stages >= 0 and capacity >= 1")
    sa, sb, sm = [], [], []

    def released(i):   # S_m(i - M) + T_MATH, or no constraint before the ring fills
        k = i - capacity
        return sm[k - 1] + t_math if k >= 1 else NEG_INF

    for i in range(1, n_stages + 1):
        a = 0.0 if i == 1 else max(sb[-1] + t_lb, released(i))
        b = max(a + t_la, released(i))
        m = max((sm[-1] + t_math) if sm else NEG_INF, b + t_lb)
        sa.append(a)
        sb.append(b)
        sm.append(m)
    return sa, sb, sm


def waves(m: int, n: int, t_m: int, t_n: int, n_sms: int) -> int:
    """W = ceil(ceil(M/T_M) * ceil(N/T_N) / SMs)."""
    return math.ceil(math.ceil(m / t_m) * math.ceil(n / t_n) / n_sms)


def overall_time(n_stages: int, capacity: int, t_la: float, t_lb: float, t_math: float,
                 n_waves: int, t_epilogue: float, t_init: float) -> float:
    """T = (S_m(S) + T_EPILOGUE) * W + T_INIT."""
    if n_stages == 0:
        return t_epilogue * n_waves + t_init
    sm = ws_recurrence(n_stages, capacity, t_la, t_lb, t_math)[2]
    return (sm[-1] + t_epilogue) * n_waves + t_init


def math_wait(n_stages: int, capacity: int, t_la: float, t_lb: float,
              t_math: float) -> list[float]:
    """Wait(i) of the page's second objective: how long MATH idles before
    stage i (the first stage waits for its data, S_b(1) + T_LB)."""
    _, sb, sm = ws_recurrence(n_stages, capacity, t_la, t_lb, t_math)
    out = []
    for i in range(n_stages):
        out.append(sb[0] + t_lb if i == 0 else sm[i] - (sm[i - 1] + t_math))
    return out


def two_point(size1: float, time1: float, size2: float, time2: float) -> tuple[float, float]:
    """The page's calibration: throughput = (size1 - size2) / (time1 - time2),
    startup latency = the time left at size 0.  Returns (throughput, latency)."""
    if time1 == time2:
        raise ValueError("two different times are needed")
    thr = (size1 - size2) / (time1 - time2)
    return thr, time1 - size1 / thr


@dataclass(frozen=True)
class AttentionRing:
    """Per-SM timing parameters of the attention kernel (one time unit, e.g.
    SM cycles or microseconds): t_load is the load of one K or V tile, t_block
    the consumer period of one key block, t_unit the per-unit cost the
    recurrence does not see (epilogue hand-off), t_init the per-block start."""
    t_load: float
    t_block: float
    t_unit: float = 0.0
    t_init: float = 0.0

    def sm_time(self, blocks_per_unit: list[int], ring_slots: int) -> float:
        """One persistent block running `blocks_per_unit` back to back through
        a ring of `ring_slots` K/V slots."""
        cap = max(1, ring_slots // 2)
        n = sum(blocks_per_unit)
        sm = ws_recurrence(n, cap, self.t_load, self.t_load, self.t_block)[2]
        return self.t_init + sm[-1] + self.t_block + self.t_unit * len(blocks_per_unit)

    def kernel_time(self, n_units: int, blocks_per_unit: int, ring_slots: int,
                    n_sms: int) -> float:
        """Full attention (equal units): the busiest SM's time when units are
        handed out dynamically, i.e. ceil(units / SMs) units on it."""
        per_sm = math.ceil(n_units / n_sms)
        return self.sm_time([blocks_per_unit] * per_sm, ring_slots)


def steady_period(capacity: int, t_la: float, t_lb: float, t_math: float) -> float:
    """Steady-state stage period of the recurrence: MATH-bound (T_MATH),
    load-bound (T_LA + T_LB), or ring-bound (a slot returns only after the
    stage M back has been loaded and computed: (T_LA + T_LB + T_MATH) / M)."""
    return max(t_math, t_la + t_lb, (t_la + t_lb + t_math) / capacity)


def load_time_from_ring_period(period: float, capacity: int, t_math: float) -> float:
    """Inverts the ring-bound case of steady_period: when a ring of
    `capacity` stages limits the pipeline, period = (2 t_load + T_MATH) /
    capacity, so one tile load takes (period * capacity - T_MATH) / 2 (A and
    B tiles of equal size).  Since (a + b) / M <= max(a, b) for M >= 2, only a
    one-stage ring is ever ring-bound in this model: it predicts that every
    ring of two or more stages runs at max(2 t_load, T_MATH)."""
    return (period * capacity - t_math) / 2.0
