"""Pins of the backward oracle (oracle/attn_oracle_bwd.c), CPU only.

The backward oracle writes out the chain rule of the forward definition.  It
is pinned to things other than itself:
  * central finite differences of the (already pinned) forward oracle: for a
    loss L = sum(dO * O), dL/dx computed numerically for every element of Q,
    K and V must match the oracle's dQ, dK, dV -- this checks the gradient
    against the forward definition, not against any gradient formula;
  * torch's fp64 autograd of softmax(scale Q K^T + mask) V (a library special
    case that shares no code with either side);
  * closed forms and invariants: one key; V rows all equal; the softmax shift
    invariance sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i; linearity in dO;
    causal row 0 depends on key 0 only.
"""
import numpy as np
import pytest
import torch

import oracle


def _inputs(S, D, seed, scale_k=1.0):
    rng = np.random.default_rng(seed)
    q, k, v, do = (rng.standard_normal((S, D)) for _ in range(4))
    return q, k * scale_k, v, do


def _loss(q, k, v, do, causal, scale):
    o, _ = oracle.attention(q[None], k[None], v[None], causal, scale)
    return float((o[0] * do).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,D", [(1, 3), (4, 3), (7, 5)])
def test_matches_finite_differences_of_the_forward(S, D, causal):
    q, k, v, do = _inputs(S, D, 10 * S + D + causal)
    scale = 0.7
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)
    eps = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, causal, scale)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], do, causal, scale)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8,
                                   err_msg="d%s vs finite differences" % name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,D", [(1, 4), (3, 4), (17, 8), (64, 16)])
def test_matches_torch_autograd_fp64(S, D, causal):
    q, k, v, do = _inputs(S, D, 100 + S, scale_k=2.0)
    scale = 1.0 / np.sqrt(D)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    s = scale * tq @ tk.T
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.tensor(do))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)
    for name, got, ref in (("dq", dq, tq.grad), ("dk", dk, tk.grad), ("dv", dv, tv.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def test_one_key():
    # S = 1: p = 1, so dV = dO and dS = p (dP - delta) = 0: dQ = dK = 0
    q, k, v, do = _inputs(1, 6, 3)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, False, 0.9)
    np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15


def test_equal_value_rows_have_no_score_gradient():
    # every row of V equal: O does not depend on the scores, so dQ = dK = 0
    # and dV_j = sum_i p_ij dO_i sums to sum_i dO_i
    q, k, _, do = _inputs(9, 4, 5)
    v = np.tile(np.array([[0.3, -1.0, 2.0, 0.5]]), (9, 1))
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, 0.5)
        assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
        np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_invariants(causal):
    q, k, v, do = _inputs(12, 5, 21)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, 0.4)
    # adding a constant to every logit of a row changes nothing: sum_j dS_ij = 0,
    # hence sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # each softmax row sums to one: sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


def test_linear_in_dout():
    q, k, v, do = _inputs(10, 4, 8)
    do2 = np.random.default_rng(9).standard_normal(do.shape)
    g1 = oracle.attention_bwd(q, k, v, do, True, 0.6)
    g2 = oracle.attention_bwd(q, k, v, do2, True, 0.6)
    g3 = oracle.attention_bwd(q, k, v, 2 * do - 3 * do2, True, 0.6)
    for a, b, c in zip(g1, g2, g3):
        np.testing.assert_allclose(c, 2 * a - 3 * b, atol=1e-12)


def test_causal_row_zero_sees_key_zero_only():
    # dO nonzero in row 0 only: under the causal mask only key 0 and value 0
    # receive gradient, and dQ_0 = 0 (a single visible key)
    q, k, v, _ = _inputs(6, 4, 13)
    do = np.zeros((6, 4))
    do[0] = [1.0, -2.0, 0.5, 3.0]
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, 0.8)
    np.testing.assert_allclose(dv[0], do[0], atol=1e-15)
    assert np.abs(dv[1:]).max() == 0 and np.abs(dk).max() < 1e-15 and np.abs(dq).max() < 1e-15


def test_batched_slices_are_independent():
    rng = np.random.default_rng(4)
    q, k, v, do = (rng.standard_normal((2, 3, 8, 4)) for _ in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, 0.5)
    b, h = 1, 2
    g = oracle.attention_bwd(q[b, h], k[b, h], v[b, h], do[b, h], True, 0.5)
    for full, one in zip((dq, dk, dv), g):
        np.testing.assert_array_equal(full[b, h], one)
