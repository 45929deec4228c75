"""CPU pins of the warp-specialization pipeline model
(warp_specialized_attention_gb300/ring_model.py, after "A Performance Model
for Warp Specialization Kernels", core formulas).  The page's worked timing
table cannot pin it (its throughput units are garbled, and its four printed
predictions imply inconsistent startup latencies), so the recurrence is held
to what the mathematics fixes: closed forms of its special cases, the
steady-state period (the max-plus cycle mean), monotonicity in the ring
depth, the wave count and the two-point calibration."""
import math
import random

import pytest

from warp_specialized_attention_gb300 import ring_model as rm


def test_free_loads_give_back_to_back_math():
    # T_LA = T_LB = 0: MATH never waits, S_m(i) = (i-1) T_MATH
    sm = rm.ws_recurrence(10, 2, 0.0, 0.0, 3.0)[2]
    assert sm == [3.0 * i for i in range(10)]


def test_single_buffer_serialises_everything():
    # M = 1: load A, load B and MATH of a stage run one after the other
    la, lb, m = 2.0, 3.0, 7.0
    sa, sb, sm = rm.ws_recurrence(6, 1, la, lb, m)
    period = la + lb + m
    assert sm == [la + lb + i * period for i in range(6)]
    assert sa == [i * period for i in range(6)]
    assert sb == [la + i * period for i in range(6)]


def test_unbounded_ring_is_a_two_server_tandem_line():
    # M >= S: loads run back to back; MATH of stage i starts at
    # max over k <= i of (k (T_LA + T_LB) + (i - k) T_MATH)
    rng = random.Random(3)
    for _ in range(20):
        la, lb, m = (rng.uniform(0.1, 5) for _ in range(3))
        n = 12
        sa, sb, sm = rm.ws_recurrence(n, n, la, lb, m)
        for i in range(1, n + 1):
            assert sa[i - 1] == pytest.approx((i - 1) * (la + lb))
            expect = max(k * (la + lb) + (i - k) * m for k in range(1, i + 1))
            assert sm[i - 1] == pytest.approx(expect)


@pytest.mark.parametrize("seed", range(8))
def test_long_run_period_is_the_cycle_mean(seed):
    rng = random.Random(seed)
    la, lb, m = (rng.uniform(0.1, 5) for _ in range(3))
    cap = rng.randint(1, 5)
    sm = rm.ws_recurrence(400, cap, la, lb, m)[2]
    measured = (sm[-1] - sm[-101]) / 100
    assert measured == pytest.approx(rm.steady_period(cap, la, lb, m), rel=1e-9)


def test_a_deeper_ring_is_never_slower():
    rng = random.Random(11)
    for _ in range(30):
        la, lb, m = (rng.uniform(0.1, 5) for _ in range(3))
        ends = [rm.ws_recurrence(40, cap, la, lb, m)[2][-1] for cap in range(1, 8)]
        assert all(a >= b - 1e-12 for a, b in zip(ends, ends[1:]))


def test_math_waits_account_for_the_whole_math_timeline():
    # S_m(S) = sum of Wait(i) + (S - 1) T_MATH
    la, lb, m, n = 1.5, 2.5, 2.0, 9
    for cap in (1, 2, 3, 9):
        sm = rm.ws_recurrence(n, cap, la, lb, m)[2]
        assert sum(rm.math_wait(n, cap, la, lb, m)) + (n - 1) * m == pytest.approx(sm[-1])


def test_waves_and_overall_time():
    assert rm.waves(1024, 1024, 128, 64, 84) == 2        # 128 tiles on 84 SMs
    assert rm.waves(512, 1024, 128, 64, 84) == 1         # 64 tiles
    assert rm.waves(1000, 1000, 128, 128, 64) == 1       # ceil(1000/128) = 8: 64 tiles
    assert rm.waves(1025, 1000, 128, 128, 64) == 2       # 9 x 8 = 72 tiles
    # T = (S_m(S) + T_EPI) W + T_INIT
    sm = rm.ws_recurrence(16, 4, 1.0, 1.0, 3.0)[2]
    assert rm.overall_time(16, 4, 1.0, 1.0, 3.0, 2, 0.5, 1.7) == pytest.approx(
        (sm[-1] + 0.5) * 2 + 1.7)


def test_two_point_calibration_recovers_a_linear_cost():
    thr, lat = 24.61, 0.77
    t = lambda size: size / thr + lat  # noqa: E731
    got_thr, got_lat = rm.two_point(128 * 64, t(128 * 64), 64 * 64, t(64 * 64))
    assert got_thr == pytest.approx(thr) and got_lat == pytest.approx(lat)


def test_ring_bound_inversion():
    # (T_LA + T_LB + T_MATH) / M never exceeds max(T_LA + T_LB, T_MATH) once
    # M >= 2, so only a one-stage ring is ever ring-bound in this model
    rng = random.Random(5)
    for _ in range(50):
        la, m = rng.uniform(0.1, 5), rng.uniform(0.1, 5)
        for cap in (2, 3, 4):
            assert rm.steady_period(cap, la, la, m) == pytest.approx(max(2 * la, m))
    t_load, t_math = 5.0, 4.0
    period = rm.steady_period(1, t_load, t_load, t_math)
    assert period == pytest.approx(2 * t_load + t_math)
    assert rm.load_time_from_ring_period(period, 1, t_math) == pytest.approx(t_load)


def test_attention_ring_adaptation():
    ring = rm.AttentionRing(t_load=1.0, t_block=3.0, t_unit=0.5, t_init=2.0)
    # MATH-bound ring: an SM's time is its blocks' MATH plus the first loads
    n_units, blocks = 300, 8
    per_sm = math.ceil(n_units / 152)
    t = ring.kernel_time(n_units, blocks, ring_slots=8, n_sms=152)
    assert t == pytest.approx(2.0 + 2 * 1.0 + per_sm * blocks * 3.0 + per_sm * 0.5)
    # two slots (one stage) serialise load and MATH
    t1 = ring.sm_time([4], ring_slots=2)
    assert t1 == pytest.approx(2.0 + 2.0 + 3 * (2 + 3.0) + 3.0 + 0.5)
