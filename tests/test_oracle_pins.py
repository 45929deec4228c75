"""Pins for the fp64 oracle: closed forms, invariants, a library special case,
hand-worked golden cases and a high-precision brute force on tiny inputs.

The attention being pinned is the Q K^T -> softmax -> P V loop of "Tawa:
Automatic Warp Specialization for Modern GPUs with Asynchronous References",
Section III-D, Algorithm 1, with the textbook softmax definition, the optional
causal mask (key j visible to query i iff j <= i) and the natural log-sum-exp
of the scaled logits.  Each pin is chosen so that a plausible slip in the oracle
(a dropped scale, the mask off by one or reversed, log2 instead of ln, a
transposed operand, a missing max subtraction) fails at least one of them.
"""
import decimal
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _eval(expr):
    """Evaluate a fixture expression: rationals, +,-,*,/ and ln()."""
    return float(eval(expr, {"__builtins__": {}}, {"ln": math.log}))


# ---------------------------------------------------------------------------
# golden: hand-derived cases


def _golden_cases():
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_hand_worked(case):
    q = np.array([[_eval(x) for x in r] for r in case["q"]])
    k = np.array([[_eval(x) for x in r] for r in case["k"]])
    v = np.array([[_eval(x) for x in r] for r in case["v"]])
    o_ref = np.array([[_eval(x) for x in r] for r in case["o"]])
    lse_ref = np.array([_eval(x) for x in case["lse"]])
    o, lse = oracle.attention(q, k, v, case["causal"], _eval(case["scale"]))
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    r = _rng(1)
    S, D = 37, 16
    q, k = r.standard_normal((S, D)), r.standard_normal((S, D))
    c = r.standard_normal(D)
    v = np.tile(c, (S, 1))
    o, _ = oracle.attention(q, k, v, causal, 0.3)
    np.testing.assert_allclose(o, v, rtol=0, atol=TOL)


def test_zero_q_unmasked_is_column_mean_and_ln_s():
    r = _rng(2)
    S, D = 50, 8
    q = np.zeros((S, D))
    k, v = r.standard_normal((S, D)), r.standard_normal((S, D))
    o, lse = oracle.attention(q, k, v, False, 0.125)
    np.testing.assert_allclose(o, np.tile(v.mean(axis=0), (S, 1)), rtol=0, atol=TOL)
    np.testing.assert_allclose(lse, np.full(S, math.log(S)), rtol=0, atol=TOL)


def test_zero_q_causal_is_prefix_mean_and_ln_count():
    r = _rng(3)
    S, D = 41, 8
    q = np.zeros((S, D))
    k, v = r.standard_normal((S, D)), r.standard_normal((S, D))
    o, lse = oracle.attention(q, k, v, True, 0.125)
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(o, prefix_mean, rtol=0, atol=TOL)
    np.testing.assert_allclose(lse, np.log(np.arange(1, S + 1)), rtol=0, atol=TOL)


def test_causal_row0_is_v0_and_scaled_dot():
    r = _rng(4)
    S, D = 9, 5
    q, k, v = (r.standard_normal((S, D)) for _ in range(3))
    scale = 0.7
    o, lse = oracle.attention(q, k, v, True, scale)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=TOL)
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < TOL


@pytest.mark.parametrize("causal", [False, True])
def test_single_key(causal):
    r = _rng(5)
    q, k, v = (r.standard_normal((1, 7)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, causal, 2.5)
    np.testing.assert_allclose(o, v, rtol=0, atol=TOL)
    assert abs(lse[0] - 2.5 * float(q[0] @ k[0])) < TOL


# ---------------------------------------------------------------------------
# invariants


@pytest.mark.parametrize("causal", [False, True])
def test_weights_sum_to_one_via_lse(causal):
    """sum_j exp(scale*q_i.k_j - LSE_i) over visible j equals 1 (the softmax
    normaliser and the reported LSE agree), and V = ones gives O = 1."""
    r = _rng(6)
    S, D = 33, 12
    q, k = r.standard_normal((S, D)), r.standard_normal((S, D))
    scale = 0.4
    o, lse = oracle.attention(q, k, np.ones((S, D)), causal, scale)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=TOL)
    logits = scale * (q @ k.T)
    for i in range(S):
        n = i + 1 if causal else S
        assert abs(np.exp(logits[i, :n] - lse[i]).sum() - 1.0) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_linear_in_v(causal):
    r = _rng(7)
    S, D = 29, 6
    q, k, v1, v2 = (r.standard_normal((S, D)) for _ in range(4))
    o1, l1 = oracle.attention(q, k, v1, causal, 0.5)
    o2, l2 = oracle.attention(q, k, v2, causal, 0.5)
    o3, l3 = oracle.attention(q, k, 2.0 * v1 - 3.0 * v2, causal, 0.5)
    np.testing.assert_allclose(o3, 2.0 * o1 - 3.0 * o2, rtol=0, atol=1e-11)
    np.testing.assert_allclose(l3, l1, rtol=0, atol=TOL)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=TOL)


def test_unmasked_invariant_under_joint_kv_permutation():
    r = _rng(8)
    S, D = 31, 10
    q, k, v = (r.standard_normal((S, D)) for _ in range(3))
    perm = r.permutation(S)
    o, lse = oracle.attention(q, k, v, False, 0.3)
    o_p, lse_p = oracle.attention(q, k[perm], v[perm], False, 0.3)
    np.testing.assert_allclose(o_p, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_p, lse, rtol=0, atol=1e-12)


def test_causal_row_ignores_later_keys():
    """Row i under the mask must not change when rows j > i of K and V do."""
    r = _rng(9)
    S, D = 24, 8
    q, k, v = (r.standard_normal((S, D)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, True, 0.35)
    for i in (0, 5, 17):
        k2, v2 = k.copy(), v.copy()
        k2[i + 1:] = r.standard_normal((S - i - 1, D)) * 10
        v2[i + 1:] = r.standard_normal((S - i - 1, D)) * 10
        o2, lse2 = oracle.attention(q, k2, v2, True, 0.35)
        np.testing.assert_allclose(o2[: i + 1], o[: i + 1], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse2[: i + 1], lse[: i + 1], rtol=0, atol=TOL)
    # ... and the last row under the mask sees every key, like the unmasked row
    o_u, lse_u = oracle.attention(q, k, v, False, 0.35)
    np.testing.assert_allclose(o[-1], o_u[-1], rtol=0, atol=TOL)
    assert abs(lse[-1] - lse_u[-1]) < TOL


def test_one_hot_limit_selects_v_row():
    """K rows are large multiples of distinct basis vectors and each query is a
    basis vector: the softmax concentrates on one key, so O picks one V row and
    LSE tends to the selected logit."""
    S = D = 16
    r = _rng(10)
    perm = r.permutation(S)
    k = 60.0 * np.eye(D)[perm]            # key j points along axis perm[j]
    target = r.permutation(S)             # query i wants key target[i]
    q = np.eye(D)[perm[target]]
    v = r.standard_normal((S, D))
    o, lse = oracle.attention(q, k, v, False, 1.0)
    np.testing.assert_allclose(o, v[target], rtol=0, atol=np.abs(v).max() * S * math.exp(-60))
    np.testing.assert_allclose(lse, 60.0, rtol=0, atol=S * math.exp(-60))


def test_scale_and_query_trade_off():
    """scale * (a q) . k == (a scale) * q . k: only the product matters."""
    r = _rng(11)
    q, k, v = (r.standard_normal((19, 9)) for _ in range(3))
    o1, l1 = oracle.attention(q * 4.0, k, v, True, 0.125)
    o2, l2 = oracle.attention(q, k, v, True, 0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# library special case: torch fp64 softmax / logsumexp on the same logits


@pytest.mark.parametrize("S", [1, 2, 3, 17, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_fp64_softmax(S, causal):
    g = torch.Generator().manual_seed(100 + S)
    D = 64 if S >= 128 else 5
    q, k, v = (torch.randn(2, S, D, generator=g, dtype=torch.float64) for _ in range(3))
    scale = 1.0 / math.sqrt(D)
    logits = scale * q @ k.transpose(-1, -2)
    if causal:
        mask = torch.ones(S, S, dtype=torch.bool).triu(1)
        logits = logits.masked_fill(mask, float("-inf"))
    o_ref = torch.softmax(logits, dim=-1) @ v
    lse_ref = torch.logsumexp(logits, dim=-1)
    o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal, scale)
    np.testing.assert_allclose(o, o_ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# brute force at 40 significant digits, no max subtraction, tiny S


@pytest.mark.parametrize("causal", [False, True])
def test_high_precision_brute_force(causal):
    ctx = decimal.Context(prec=40)
    r = _rng(12)
    S, D = 3, 4
    q, k, v = (r.standard_normal((S, D)) for _ in range(3))
    scale = 0.6
    o, lse = oracle.attention(q, k, v, causal, scale)
    Dec = decimal.Decimal
    for i in range(S):
        keys = range(i + 1) if causal else range(S)
        w = {}
        for j in keys:
            dot = sum((Dec(float(q[i, d])) * Dec(float(k[j, d])) for d in range(D)), Dec(0))
            w[j] = ctx.exp(ctx.multiply(Dec(scale), dot))
        z = sum(w.values(), Dec(0))
        assert abs(float(ctx.ln(z)) - lse[i]) < 1e-13
        for d in range(D):
            num = sum((w[j] * Dec(float(v[j, d])) for j in keys), Dec(0))
            assert abs(float(num / z) - o[i, d]) < 1e-13


# ---------------------------------------------------------------------------
# API consistency


def test_rows_entry_matches_full():
    r = _rng(13)
    S, D = 40, 8
    q, k, v = (r.standard_normal((S, D)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, True, 0.2)
    rows = np.array([39, 0, 17, 17, 3])
    o_r, lse_r = oracle.attention_rows(q[rows], k, v, rows, True, 0.2)
    np.testing.assert_array_equal(o_r, o[rows])
    np.testing.assert_array_equal(lse_r, lse[rows])


def test_rows_out_of_range_rejected():
    q = np.zeros((1, 4))
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, np.zeros((3, 4)), np.zeros((3, 4)), [3], False, 1.0)


def test_batched_heads_independent():
    r = _rng(14)
    q, k, v = (r.standard_normal((2, 3, 12, 4)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, True, 0.5)
    for b in range(2):
        for h in range(3):
            o1, l1 = oracle.attention(q[b, h], k[b, h], v[b, h], True, 0.5)
            np.testing.assert_array_equal(o[b, h], o1)
            np.testing.assert_array_equal(lse[b, h], l1)
