"""GPU parity of the E4M3 path of fmha_fwd (through the C ABI) against the fp64
CPU oracle, on the same E4M3 values.

The bound comes from the arithmetic.  Both sides see identical E4M3 inputs.
Q K^T is exact in fp32: E4M3 products are exact and 128 of them sum with fp32
rounding only.  LSE comes from the fp32 sum of the unrounded exponentials, so
it keeps the 16-bit bar, |dLSE| <= 1e-3.

O differs from the definition because P is rounded to E4M3 before P V.  With
lazy-rescale threshold tau the kernel's running maximum m_K is within tau of
the true one, and it stores p' = 2^(8 - tau) * exp2(s*c - m_K) <= 256.  A
normal E4M3 p' (>= 2^-6) is off by at most 2^-4 relative (3 mantissa bits,
round to nearest).  A smaller p' is off by at most 2^-10 absolute, which is at
most 2^(-18 + tau) in units of the row's true maximum.  With p_j = exp(s_j -
s_max) and l = sum_j p_j = exp(LSE - s_max):

    |dO_id| <= 2^-4 * sum_j p_j |v_jd| / l  +  2^(-18+tau) * sum_j |v_jd| / l
               + 2^-8 * |O_id| (bf16 output)  + 1e-4 (fp32, ex2)

where sum_j p_j |v_jd| / l is attention with |V| in place of V, which the
oracle computes; s_max (the row's largest visible logit) comes from an fp64
product in the test.  That bound holds element by element.  Rounding to nearest
is unbiased, so the errors of many keys should also add up like independent
ones.  Their expected square is at most (2^-4)^2/3 * sum_j p_j^2 v_jd^2 / l^2
= (2^-4)^2/3 * A2_id * exp(LSE2_i - 2 LSE_i), where A2 and LSE2 are the
oracle's attention of V^2 at twice the scale (plus the subnormal term's
square, (2^(-18+tau))^2/3 * sum_j v_jd^2 / l^2).  The root mean square of the
error over all compared elements must stay within 3x that (plus the bf16
term): a biased or misplaced P fails it long before the hard bound.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic
import warp_specialized_attention_gb300 as wsa

pytestmark = pytest.mark.gpu

TOL_LSE = 1e-3
U8 = 2.0 ** -4      # E4M3 unit roundoff
U_BF16 = 2.0 ** -8


def _gpu(q, k, v, causal, scale):
    qd, kd, vtd = q.cuda(), k.cuda(), synthetic.kernel_v(v).cuda()
    o = torch.full(q.shape, float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full(q.shape[:3], float("nan"), device="cuda", dtype=torch.float32)
    wsa.fmha_fwd(qd, kd, vtd, o, lse, causal=causal, scale=scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def _bounds(q64, k64, v64, rows, causal, scale, o_ref, lse_ref, tau):
    """Per-element hard bound and expected square of the error (see the module
    docstring): oracle calls, plus s_max and the key sums of |V| and V^2."""
    o_abs, _ = oracle.attention_rows(q64, k64, np.abs(v64), rows, causal, scale)
    a2, lse2 = oracle.attention_rows(q64, k64, v64 ** 2, rows, causal, 2 * scale)
    s = (q64 @ k64.T) * scale
    vis = (np.arange(k64.shape[0])[None, :] <= rows[:, None]) if causal else \
        np.ones(s.shape, dtype=bool)
    s_max = np.where(vis, s, -np.inf).max(axis=1)
    inv_l = np.exp(s_max - lse_ref)[:, None]                 # 1 / l
    sum_abs_v = vis.astype(np.float64) @ np.abs(v64)         # sum over visible keys
    sum_v2 = vis.astype(np.float64) @ (v64 ** 2)
    sub = 2.0 ** (-18 + tau)
    hard = U8 * o_abs + sub * sum_abs_v * inv_l + U_BF16 * np.abs(o_ref) + 1e-4
    msq = (U8 ** 2 / 3 * a2 * np.exp(lse2 - 2 * lse_ref)[:, None]
           + sub ** 2 / 3 * sum_v2 * inv_l ** 2)
    return hard, msq


def _check(o, lse, q, k, v, bh_rows, causal, scale, label, tau=8.0):
    """Compare selected rows of the given (b, h) slices; returns worst errors."""
    worst = {"o": 0.0, "lse": 0.0, "rms": 0.0, "rms_bound": 0.0}
    sq_err = sq_bound = 0.0
    count = 0
    for (b, h), rows in bh_rows:
        q64, k64, v64 = (t[b, h].double().numpy() for t in (q, k, v))
        o_ref, lse_ref = oracle.attention_rows(q64[rows], k64, v64, rows, causal, scale)
        hard, msq = _bounds(q64[rows], k64, v64, rows, causal, scale, o_ref, lse_ref, tau)
        d_o = np.abs(o[b, h, rows] - o_ref)
        d_l = np.abs(lse[b, h, rows] - lse_ref)
        assert np.isfinite(o[b, h, rows]).all() and np.isfinite(lse[b, h, rows]).all()
        ratio = (d_o / hard).max()
        assert ratio <= 1.0, "%s: O error %.3e exceeds the E4M3 bound (ratio %.2f)" % (
            label, d_o.max(), ratio)
        worst["o"] = max(worst["o"], float(d_o.max()))
        worst["lse"] = max(worst["lse"], float(d_l.max()))
        sq_err += float((d_o ** 2).sum())
        sq_bound += float((msq + (U_BF16 * np.abs(o_ref)) ** 2).sum())
        count += d_o.size
    rms, rms_bound = math.sqrt(sq_err / count), 3 * math.sqrt(sq_bound / count)
    print("PARITY-E4M3 %s max_err_O %.3e rms_err_O %.3e (rms bound %.3e) max_err_LSE %.3e"
          % (label, worst["o"], rms, rms_bound, worst["lse"]))
    assert worst["lse"] <= TOL_LSE, "%s: LSE error %g" % (label, worst["lse"])
    assert rms <= rms_bound, "%s: O errors do not behave like roundings (rms %.3e > %.3e)" % (
        label, rms, rms_bound)


SMALL = [
    # B, H, S, causal, k_mult
    (1, 2, 256, False, 1.0),
    (1, 1, 128, True, 1.0),
    (2, 3, 384, True, 1.0),
    (1, 2, 1008, False, 1.0),     # ragged last key block (S % 128 = 112)
    (1, 1, 16, True, 1.0),        # one partial block
    (1, 1, 2048, False, 1.0),
    (1, 2, 784, True, 4.0),       # sharpened logits, ragged
    (3, 2, 1536, True, 1.0),      # several units per block on most SMs
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B%dH%dS%d-%s-k%g" % (
    c[0], c[1], c[2], "causal" if c[3] else "full", c[4]))
def test_e4m3_small_full_compare(case):
    B, H, S, causal, k_mult = case
    w = synthetic.Workload("e4m3", B, H, S, 128, "e4m3", causal, k_mult, 7000 + S)
    q, k, v = synthetic.make_inputs(w)
    o, lse = _gpu(q, k, v, causal, w.scale)
    rows = np.arange(S, dtype=np.int64)
    _check(o, lse, q, k, v, [((b, h), rows) for b in range(B) for h in range(H)], causal,
           w.scale, w.describe())


@pytest.mark.parametrize("w", synthetic.FP8_WORKLOADS, ids=lambda w: w.name)
def test_e4m3_named_workload_sampled(w):
    q, k, v = synthetic.make_inputs(w)
    o, lse = _gpu(q, k, v, w.causal, w.scale)
    rng = np.random.default_rng(w.seed)
    BH = w.B * w.H
    picks = []
    for bh in sorted({0, BH // 2, BH - 1}):
        rows = {0, 1, 127, 128, w.S - 1} | set(rng.integers(0, w.S, size=24).tolist())
        picks.append((divmod(bh, w.H), np.array(sorted(rows), dtype=np.int64)))
    _check(o, lse, q, k, v, picks, w.causal, w.scale, w.describe() + " (sampled rows)")


def test_e4m3_causal_4k_sampled():
    """E4M3 at B4 H32 S4096 causal: 2048 units handed out longest first in
    head groups, so most blocks run a dozen units of different lengths;
    sampled rows of three slices against the oracle, and no device-side
    wait may give up."""
    w = synthetic.Workload("e4m3-causal-4k", 4, 32, 4096, 128, "e4m3", True, 1.0, 7104)
    q, k, v = synthetic.make_inputs(w)
    o, lse = _gpu(q, k, v, w.causal, w.scale)
    rng = np.random.default_rng(w.seed)
    picks = []
    for bh in (0, 64, 127):
        rows = {0, 1, 127, 128, 255, 256, w.S - 1} | set(rng.integers(0, w.S, size=24).tolist())
        picks.append((divmod(bh, w.H), np.array(sorted(rows), dtype=np.int64)))
    _check(o, lse, q, k, v, picks, w.causal, w.scale, w.describe() + " (sampled rows)")


def test_e4m3_threshold_knob():
    """The E4M3 threshold may be set anywhere in [0, 8] (P then stored as
    2^(8-tau) P; 8 is the default): the result must stay within the bounds."""
    w = synthetic.Workload("e4m3-tau", 1, 2, 1024, 128, "e4m3", True, 1.0, 77)
    q, k, v = synthetic.make_inputs(w)
    qd, kd, vtd = q.cuda(), k.cuda(), synthetic.kernel_v(v).cuda()
    for tau in (0.0, 4.0, 8.0):
        o = torch.full(q.shape, float("nan"), device="cuda", dtype=torch.bfloat16)
        lse = torch.full(q.shape[:3], float("nan"), device="cuda", dtype=torch.float32)
        assert wsa.fmha_fwd_testing(qd, kd, vtd, o, lse, True, w.scale, 0, 1.0, tau) == wsa.FMHA_OK
        assert wsa.get_device_status() == wsa.FMHA_OK
        rows = np.arange(w.S, dtype=np.int64)
        _check(o.cpu().double().numpy(), lse.cpu().double().numpy(), q, k, v,
               [((0, h), rows) for h in range(2)], True, w.scale,
               "%s tau=%g" % (w.describe(), tau), tau=tau)
