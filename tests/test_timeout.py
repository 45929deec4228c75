"""Failure detection without a GPU fault: every mbarrier wait in the kernel is
bounded.  The test hook drops the first "P ready" arrival of query tile 0, so
the MMA issuer's wait runs out; the block must then drain its copies and MMAs,
free Tensor Memory, and exit, the host must read FMHA_ERR_TIMEOUT from the
status word, and the context must stay usable for the next call."""
import time

import numpy as np
import pytest
import torch

import oracle
import synthetic
import warp_specialized_attention_gb300 as wsa

pytestmark = pytest.mark.gpu


def _inputs():
    w = synthetic.Workload("timeout", 1, 2, 512, 128, "f16", False, 1.0, 31)
    q, k, v = synthetic.make_inputs(w)
    return w, q, k, v


def test_hook_without_fault_matches_fmha_fwd():
    w, q, k, v = _inputs()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = wsa.attention(qd, kd, vd, causal=False, scale=w.scale)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    assert wsa.fmha_fwd_testing(qd, kd, vd, o2, l2, False, w.scale, 0, 1.0) == wsa.FMHA_OK
    assert wsa.get_device_status() == wsa.FMHA_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_dropped_arrival_times_out_and_context_survives():
    w, q, k, v = _inputs()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], device="cuda", dtype=torch.float32)
    assert wsa.get_device_status() == wsa.FMHA_OK
    t0 = time.time()
    assert wsa.fmha_fwd_testing(qd, kd, vd, o, lse, False, w.scale, 1, 0.25) == wsa.FMHA_OK
    assert wsa.get_device_status() == wsa.FMHA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    # the status word was cleared and the context still works
    assert wsa.get_device_status() == wsa.FMHA_OK
    o2, lse2 = wsa.attention(qd, kd, vd, causal=False, scale=w.scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    o_ref, lse_ref = oracle.attention(q.double().numpy(), k.double().numpy(),
                                      v.double().numpy(), False, w.scale)
    assert np.abs(o2.cpu().double().numpy() - o_ref).max() <= 1e-2
    assert np.abs(lse2.cpu().double().numpy() - lse_ref).max() <= 1e-3
