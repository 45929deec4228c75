"""GPU check of fmha_bwd_noalloc, the allocation-free backward entry point (its
scratch is a device array of the library).  Collected last on purpose: it must
pass both alone and after every other test has run in the same process.

Two calls in a row must give what fmha_bwd (caller workspace) gives on the
same inputs: dK and dV bit for bit (no atomics), dQ to within the reordering
of its fp32 atomic additions.  The second call checks that the shared scratch
is cleared between calls (dQ is accumulated in it).
"""
import pytest
import torch

import synthetic
import warp_specialized_attention_gb300 as wsa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    (1, 2, 1000, 128, "f16", True),
    (2, 2, 768, 64, "bf16", False),
], ids=lambda c: "B%dH%dS%dD%d-%s-%s" % (c[0], c[1], c[2], c[3], c[4],
                                       "causal" if c[5] else "full"))
def test_noalloc_matches_workspace_entry_two_calls_in_a_row(case):
    B, H, S, D, dt, causal = case
    w = synthetic.Workload("noalloc", B, H, S, D, dt, causal, 1.0, 6100 + S)
    q, k, v = (t.cuda() for t in synthetic.make_inputs(w))
    g = torch.Generator().manual_seed(w.seed + 1)
    d_o = torch.randn(q.shape, generator=g).to(q.dtype).cuda()
    o, lse = wsa.attention(q, k, v, causal=causal, scale=w.scale)
    ref = wsa.attention_backward(q, k, v, o, lse, d_o, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        wsa.fmha_bwd_noalloc(q, k, v, o, lse, d_o, dq, dk, dv, causal=causal, scale=w.scale)
        assert wsa.get_device_status() == wsa.FMHA_OK
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), "call %d" % call
        tol = 1e-3 * ref[0].float().abs().max().item() + 1e-6
        err = (dq.float() - ref[0].float()).abs().max().item()
        assert err <= tol, "call %d: dQ differs by %g" % (call, err)
