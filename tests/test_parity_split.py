"""GPU parity of key-split units (full attention, head dim 128) against the
fp64 CPU oracle, through the C ABI.

fmha_fwd splits the units of a short last wave: each becomes two 128-row
halves whose two query tiles take half of the key blocks each, and tile 0
merges the two partial results in the block.  The merge is the online
softmax's own rescaling applied once more: with per-tile running maxima m_t
and sums l_t, the row's statistics are m = max(m_0, m_1) and
l = l_0 2^(m_0 - m) + l_1 2^(m_1 - m), and O is the two tiles' O weighted by
2^(m_t - m) / l.  These tests fix the number of split units
(fmha_fwd_split_testing) and compare every mix -- none, some, all -- element
by element with the oracle at the bar of the other parity tests
(|dO| <= 1e-2, |dLSE| <= 1e-3; E4M3 against its derived bound).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import warp_specialized_attention_gb300 as wsa
from test_parity import stratified_rows
from test_parity_fp8 import _check as _check_e4m3

pytestmark = pytest.mark.gpu

TOL_O = 1e-2
TOL_LSE = 1e-3


def _run(qd, kd, vd, scale, split_units, out_dtype):
    o = torch.full(qd.shape, float("nan"), device="cuda", dtype=out_dtype)
    lse = torch.full(qd.shape[:3], float("nan"), device="cuda", dtype=torch.float32)
    st = wsa.fmha_fwd_split_testing(qd, kd, vd, o, lse, False, scale, split_units)
    assert st == wsa.FMHA_OK, st
    assert wsa.get_device_status() == wsa.FMHA_OK
    return o, lse


CASES = [
    # B, H, S, dtype, k_mult, split-unit counts (units = B * H * ceil(S / 256))
    (1, 2, 1024, "f16", 1.0, (0, 1, 3, 8)),
    (2, 3, 1000, "bf16", 1.0, (0, 5, 24)),     # ragged: the last key block is partial
    (1, 1, 256, "f16", 1.0, (1,)),             # one key block per tile
    (1, 2, 2048, "f16", 4.0, (16,)),           # sharpened logits: maxima raised mid-unit
    (1, 1, 8192, "bf16", 1.0, (0, 32)),        # 32 key blocks per tile
    (1, 2, 1152 + 128, "bf16", 1.0, (2, 10)),  # S = 1280: 5 query blocks, 10 key blocks
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dS%d-%s-k%g" % c[:5])
def test_key_split_mixes_match_the_oracle(case):
    B, H, S, dt, k_mult, splits = case
    w = synthetic.Workload("split", B, H, S, 128, dt, False, k_mult, 9100 + S + B)
    q, k, v = synthetic.make_inputs(w)
    o_ref, lse_ref = oracle.attention(q.double().numpy(), k.double().numpy(),
                                      v.double().numpy(), False, w.scale)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for n in splits:
        o, lse = _run(qd, kd, vd, w.scale, n, qd.dtype)
        og, lg = o.cpu().double().numpy(), lse.cpu().double().numpy()
        assert np.isfinite(og).all() and np.isfinite(lg).all(), "non-finite output"
        eo, el = float(np.abs(og - o_ref).max()), float(np.abs(lg - lse_ref).max())
        print("PARITY-SPLIT %s split_units=%d max_err_O %.3e max_err_LSE %.3e"
              % (w.describe(), n, eo, el))
        assert eo <= TOL_O and el <= TOL_LSE, "split %d: max err O %g LSE %g" % (n, eo, el)


def test_key_split_is_deterministic():
    """The merge does not depend on which tile finishes first: two launches
    give the same bits."""
    w = synthetic.Workload("split-det", 1, 4, 2048, 128, "bf16", False, 1.0, 9301)
    q, k, v = synthetic.make_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = _run(qd, kd, vd, w.scale, 32, qd.dtype)
    o2, l2 = _run(qd, kd, vd, w.scale, 32, qd.dtype)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_automatic_split_matches_whole_units():
    """fmha_fwd's own choice (-1) against no split, both against the oracle,
    on a shape whose few units all get split on a GPU with 16 or more SMs."""
    w = synthetic.Workload("split-auto", 2, 2, 1024, 128, "f16", False, 1.0, 9302)
    q, k, v = synthetic.make_inputs(w)
    o_ref, lse_ref = oracle.attention(q.double().numpy(), k.double().numpy(),
                                      v.double().numpy(), False, w.scale)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for n in (-1, 0):
        o, lse = _run(qd, kd, vd, w.scale, n, qd.dtype)
        eo = float(np.abs(o.cpu().double().numpy() - o_ref).max())
        el = float(np.abs(lse.cpu().double().numpy() - lse_ref).max())
        assert eo <= TOL_O and el <= TOL_LSE, "split %d: max err O %g LSE %g" % (n, eo, el)


@pytest.mark.parametrize("S,splits", [(1024, (0, 3, 8)), (1008, (8,))], ids=["S1024", "S1008"])
def test_key_split_e4m3(S, splits):
    """E4M3 inputs (V transposed, O bf16): each tile stores its P against its
    own running maximum, so the derived E4M3 bound still holds per element."""
    w = synthetic.Workload("split-e4m3", 1, 2, S, 128, "e4m3", False, 1.0, 9400 + S)
    q, k, v = synthetic.make_inputs(w)
    qd, kd, vtd = q.cuda(), k.cuda(), synthetic.kernel_v(v).cuda()
    rows = np.arange(S, dtype=np.int64)
    for n in splits:
        o, lse = _run(qd, kd, vtd, w.scale, n, torch.bfloat16)
        _check_e4m3(o.cpu().double().numpy(), lse.cpu().double().numpy(), q, k, v,
                    [((0, h), rows) for h in range(2)], False, w.scale,
                    "%s split_units=%d" % (w.describe(), n))


def test_headline_shape_at_batch_one_with_key_split_tail():
    """B1 H32 S16384 D128 f16 through fmha_fwd: 2048 units leave a last wave of
    72 on 152 SMs, so the tail runs as 144 key-split half-units, 64 key blocks
    per tile.  Rows i = 0 (mod 8) plus the last 128 of all 32 slices against the
    oracle -- every unit contributes rows, the split ones included."""
    w = synthetic.Workload("headline-b1", 1, 32, 16384, 128, "f16", False, 1.0, 9501)
    q, k, v = synthetic.make_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = _run(qd, kd, vd, w.scale, -1, qd.dtype)
    o, lse = o.cpu(), lse.cpu()
    rows = stratified_rows(w.S)
    worst_o = worst_l = 0.0
    for h in range(w.H):
        o_ref, lse_ref = oracle.attention_rows(
            q[0, h, rows].double().numpy(), k[0, h].double().numpy(),
            v[0, h].double().numpy(), rows, False, w.scale)
        og, lg = o[0, h, rows].double().numpy(), lse[0, h, rows].double().numpy()
        assert np.isfinite(og).all() and np.isfinite(lg).all(), "non-finite output"
        worst_o = max(worst_o, float(np.abs(og - o_ref).max()))
        worst_l = max(worst_l, float(np.abs(lg - lse_ref).max()))
    print("PARITY-SPLIT %s (%d rows x %d slices) max_err_O %.3e max_err_LSE %.3e"
          % (w.describe(), rows.size, w.H, worst_o, worst_l))
    assert worst_o <= TOL_O and worst_l <= TOL_LSE, "max err O %g LSE %g" % (worst_o, worst_l)
