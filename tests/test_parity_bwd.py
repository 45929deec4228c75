"""GPU parity of fmha_bwd (through the C ABI) against the fp64 backward oracle.

The GPU's forward supplies O and LSE, as a training step would; the oracle
recomputes everything from Q, K, V and dO.  The bound comes from the kernel's
arithmetic, with u the unit roundoff of the 16-bit type (2^-11 f16, 2^-8
bf16):
  * P is rounded to 16 bits for dV += P^T dO:
        |d dV_jd| <= u sum_i P_ij |dO_id|  + u |dV_jd|      (output rounding)
  * dS = P (dP - delta) is rounded to 16 bits for dK and dQ.  delta_i = dO_i . O_i
    uses the forward's 16-bit O, which is off by at most u |O_id| plus the
    forward's own error (e_O, the 1e-2 forward bar at worst; bounded here by
    the measured |O_gpu - O_ref|):
        err_delta_i <= sum_d |dO_id| (u |O_id| + |O_gpu,id - O_ref,id|)
        |d dK_jd| <= scale sum_i (u |dS_ij| + P_ij err_delta_i) |q_id|  + u |dK_jd|
        |d dQ_id| <= scale sum_j (u |dS_ij| + P_ij err_delta_i) |k_jd|  + u |dQ_id|
  * fp32 accumulation, exp2 and the LSE of the forward (<= 1e-3 absolute,
    relative in P) add err_P = |LSE_gpu - LSE_ref| + 1e-5 relative to every P
    term, and 1e-5 of the largest magnitude.
The magnitudes |P|, |dS| in these sums are fp64 values computed in the test
from the inputs and the oracle's LSE; the expected gradients come only from
oracle.attention_bwd.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import warp_specialized_attention_gb300 as wsa

pytestmark = pytest.mark.gpu


def _u(dt):
    return 2.0 ** -8 if dt == "bf16" else 2.0 ** -11


def _run_gpu(q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = wsa.attention(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    wsa.fmha_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, causal=causal, scale=scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    return [t.cpu().double().numpy() for t in (o, lse, dq, dk, dv)]


def _bounds(q, k, v, do, o_gpu, lse_gpu, causal, scale, u):
    """Per-element bounds for dq, dk, dv of one slice (fp64 magnitudes)."""
    S = q.shape[0]
    o_ref, lse_ref = oracle.attention(q[None], k[None], v[None], causal, scale)
    o_ref, lse_ref = o_ref[0], lse_ref[0]
    s = (q @ k.T) * scale
    if causal:
        s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    p = np.exp(s - lse_ref[:, None])                       # exact softmax rows
    delta = (do * o_ref).sum(axis=1)
    ds = p * (do @ v.T - delta[:, None])
    err_delta = (np.abs(do) * (u * np.abs(o_ref) + np.abs(o_gpu - o_ref))).sum(axis=1)
    err_p = np.abs(lse_gpu - lse_ref) + 1e-5                # relative error of each P
    pe = p * (1 + err_p[:, None])
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)
    t_ds = u * np.abs(ds) + pe * err_delta[:, None] + err_p[:, None] * np.abs(ds)
    b_dv = u * (pe.T @ np.abs(do)) + err_p.max() * (p.T @ np.abs(do)) + u * np.abs(dv)
    b_dk = scale * (t_ds.T @ np.abs(q)) + u * np.abs(dk)
    b_dq = scale * (t_ds @ np.abs(k)) + u * np.abs(dq)
    return (dq, dk, dv), (b_dq, b_dk, b_dv)


def _compare(label, got, ref, bound):
    worst = 0.0
    for name, g, r, b in zip(("dQ", "dK", "dV"), got, ref, bound):
        assert np.isfinite(g).all(), "%s: non-finite %s" % (label, name)
        err = np.abs(g - r)
        lim = b + 1e-5 * np.abs(r).max() + 1e-6
        ratio = float((err / lim).max())
        worst = max(worst, ratio)
        print("PARITY-BWD %s %s max_err %.3e max|ref| %.3e (worst error/bound %.2f)"
              % (label, name, err.max(), np.abs(r).max(), ratio))
        assert ratio <= 1.0, "%s: %s error %.3e exceeds its bound" % (label, name, err.max())
    return worst


SMALL = [
    # B, H, S, D, dtype, causal
    (1, 2, 256, 64, "f16", False),
    (1, 1, 128, 128, "bf16", True),
    (2, 2, 384, 128, "f16", True),
    (1, 2, 1000, 64, "bf16", False),    # ragged last block
    (1, 1, 1, 128, "f16", False),       # one key
    (1, 1, 17, 64, "f16", True),
    (1, 1, 129, 128, "f16", True),      # one row past a block
    (1, 2, 768, 128, "bf16", True),
    (2, 1, 640, 128, "f16", False),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B%dH%dS%dD%d-%s-%s" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
def test_bwd_small_full_compare(case):
    B, H, S, D, dt, causal = case
    w = synthetic.Workload("bwd", B, H, S, D, dt, causal, 1.0, 5000 + S + D)
    q, k, v = synthetic.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    do = torch.randn(q.shape, generator=g).to(q.dtype)
    o, lse, dq, dk, dv = _run_gpu(q, k, v, do, causal, w.scale)
    for b in range(B):
        for h in range(H):
            args = [t[b, h].double().numpy() for t in (q, k, v, do)]
            ref, bound = _bounds(*args, o[b, h], lse[b, h], causal, w.scale, _u(dt))
            _compare("%s b%d h%d" % (w.describe(), b, h), (dq[b, h], dk[b, h], dv[b, h]), ref,
                     bound)


def test_bwd_bench_shape_sampled_slices():
    """The backward benchmark's shape (B4 H32 S4096 D128 bf16 causal): every
    output finite, two whole (batch, head) slices compared to the oracle."""
    w = synthetic.by_name("b4h32s4k_d128_bf16_causal")
    q, k, v = synthetic.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    do = torch.randn(q.shape, generator=g).to(q.dtype)
    o, lse, dq, dk, dv = _run_gpu(q, k, v, do, w.causal, w.scale)
    for t in (dq, dk, dv):
        assert np.isfinite(t).all()
    for bh in (0, w.B * w.H - 1):
        b, h = divmod(bh, w.H)
        args = [t[b, h].double().numpy() for t in (q, k, v, do)]
        ref, bound = _bounds(*args, o[b, h], lse[b, h], w.causal, w.scale, _u(w.dtype))
        _compare("%s slice %d" % (w.describe(), bh), (dq[b, h], dk[b, h], dv[b, h]), ref, bound)


def test_bwd_headline_shape_one_slice():
    """The backward benchmark's default shape (B4 H32 S16384 D128 f16, the
    launch bench.py times): every output finite, the last (batch, head) slice
    compared in full to the oracle (an S x S problem, a few seconds of fp64
    work on the host)."""
    w = synthetic.by_name("b4h32s16k_d128_f16")
    q, k, v = synthetic.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    do = torch.randn(q.shape, generator=g).to(q.dtype)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = wsa.attention(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    wsa.fmha_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, causal=w.causal, scale=w.scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all().item()
    b, h = w.B - 1, w.H - 1
    args = [t[b, h].double().numpy() for t in (q, k, v, do)]
    got = [t[b, h].cpu().double().numpy() for t in (dq, dk, dv)]
    ref, bound = _bounds(*args, o[b, h].cpu().double().numpy(), lse[b, h].cpu().double().numpy(),
                         w.causal, w.scale, _u(w.dtype))
    _compare("%s slice (%d, %d)" % (w.describe(), b, h), got, ref, bound)


def test_bwd_d64_sharp_causal_shape_sampled_slices():
    """B2 H16 S8192 D64 f16 causal with K scaled by 4 (logits spread four
    times wider, a sharply peaked softmax): every output finite, the first and
    last (batch, head) slices compared in full to the oracle."""
    w = synthetic.by_name("b2h16s8k_d64_f16_causal_ksharp")
    q, k, v = synthetic.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    do = torch.randn(q.shape, generator=g).to(q.dtype)
    o, lse, dq, dk, dv = _run_gpu(q, k, v, do, w.causal, w.scale)
    for t in (dq, dk, dv):
        assert np.isfinite(t).all()
    for bh in (0, w.B * w.H - 1):
        b, h = divmod(bh, w.H)
        args = [t[b, h].double().numpy() for t in (q, k, v, do)]
        ref, bound = _bounds(*args, o[b, h], lse[b, h], w.causal, w.scale, _u(w.dtype))
        _compare("%s slice %d" % (w.describe(), bh), (dq[b, h], dk[b, h], dv[b, h]), ref, bound)


def test_bwd_rejects_e4m3_and_small_workspace():
    q = torch.zeros(1, 1, 128, 128, dtype=torch.float16, device="cuda")
    o, lse = wsa.attention(q, q, q)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        wsa.fmha_bwd(q, q, q, o, lse, q, dq, dk, dv, workspace=small)


@pytest.mark.parametrize("causal,dtype", [(False, torch.float16), (True, torch.bfloat16)])
def test_autograd_wrapper_matches_the_entry_points(causal, dtype):
    """flash_attention through torch.autograd gives the outputs of attention()
    and the gradients of fmha_bwd for the incoming gradient (dK, dV bit for
    bit; dQ sums its key blocks in an unspecified order, so to 16-bit
    rounding); the entry points themselves are checked against the oracle
    above."""
    w = synthetic.Workload("autograd", 2, 3, 520, 64, "f16" if dtype == torch.float16 else "bf16",
                           causal, 1.0, 4242)
    q, k, v = (t.cuda() for t in synthetic.make_inputs(w))
    g = torch.Generator().manual_seed(7)
    d_o = torch.randn(q.shape, generator=g).to(dtype).cuda()
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = wsa.flash_attention(qa, ka, va, causal=causal, scale=w.scale)
    o.backward(d_o)
    o_ref, lse_ref = wsa.attention(q, k, v, causal=causal, scale=w.scale)
    dq_r, dk_r, dv_r = wsa.attention_backward(q, k, v, o_ref, lse_ref, d_o, causal=causal,
                                              scale=w.scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    assert torch.equal(o.detach(), o_ref)
    assert torch.equal(ka.grad, dk_r) and torch.equal(va.grad, dv_r)
    ulp = 2.0 ** -10 if dtype == torch.float16 else 2.0 ** -7
    diff = (qa.grad.float() - dq_r.float()).abs()
    assert bool((diff <= ulp * dq_r.float().abs() + 1e-5 * float(dq_r.float().abs().max())).all())


def test_autograd_lse_output_is_not_differentiable():
    """AttentionFunction returns LSE marked non-differentiable: O carries the
    graph, LSE does not, and a backward through O alone needs no check of an
    LSE gradient."""
    w = synthetic.Workload("autograd-lse", 1, 2, 256, 64, "f16", True, 1.0, 4243)
    q, k, v = (t.cuda().requires_grad_(True) for t in synthetic.make_inputs(w))
    o, lse = wsa.AttentionFunction.apply(q, k, v, True, w.scale)
    assert o.requires_grad and not lse.requires_grad
    o.float().sum().backward()
    assert wsa.get_device_status() == wsa.FMHA_OK
    for t in (q, k, v):
        assert t.grad is not None and torch.isfinite(t.grad).all().item()
