"""fmha_fwd_host: host-resident tensors, transfers overlapped with compute in
chunks of (batch, head) slices.  Rows of different slices are independent, so
the outputs must be bit-identical to fmha_fwd on the same staged inputs (the
chunks key-split the units that fmha_fwd splits on the whole problem)."""
import pytest
import torch

import synthetic
import warp_specialized_attention_gb300 as wsa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,causal,dtype,chunks", [
    ((2, 3, 384, 128), False, torch.float16, 0),
    ((2, 3, 384, 128), True, torch.bfloat16, 4),
    ((1, 5, 300, 64), True, torch.float16, 1),
    ((1, 2, 256, 64), False, torch.float16, 64),   # more chunks than slices
    ((2, 3, 512, 128), False, torch.float16, 4),    # every unit key-split
    ((1, 40, 1024, 128), False, torch.bfloat16, 3),  # the last units key-split (152 SMs)
    ((1, 40, 1024, 128), False, torch.float16, 0),
])
def test_host_entry_matches_device_entry(shape, causal, dtype, chunks):
    B, H, S, D = shape
    w = synthetic.Workload("host", B, H, S, D, "f16" if dtype == torch.float16 else "bf16",
                           causal, 1.0, 123 + S)
    q, k, v = synthetic.make_inputs(w)
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    hl = torch.full(q.shape[:3], float("nan"), dtype=torch.float32).pin_memory()
    q_dev, k_dev, v_dev, o_dev = (torch.empty(q.shape, dtype=q.dtype, device="cuda")
                                  for _ in range(4))
    lse_dev = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    wsa.fmha_fwd_host(hq, hk, hv, ho, hl, q_dev, k_dev, v_dev, o_dev, lse_dev, causal=causal,
                      scale=w.scale,
                      n_chunks=chunks)
    assert wsa.get_device_status() == wsa.FMHA_OK
    o_ref, l_ref = wsa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    assert torch.equal(ho, o_ref.cpu()) and torch.equal(hl, l_ref.cpu())


def test_host_entry_pageable_memory_and_reuse():
    w = synthetic.Workload("host2", 1, 4, 512, 128, "f16", False, 1.0, 77)
    q, k, v = synthetic.make_inputs(w)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32)
    staging = [torch.empty(q.shape, dtype=q.dtype, device="cuda") for _ in range(4)]
    lse_dev = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    o_ref, l_ref = wsa.attention(q.cuda(), k.cuda(), v.cuda(), scale=w.scale)
    for _ in range(2):  # the staging buffers and copy streams are reused
        wsa.fmha_fwd_host(q, k, v, o, lse, *staging, lse_dev, scale=w.scale, n_chunks=3)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, l_ref.cpu())


@pytest.mark.parametrize("shape,causal,dtype,chunks", [
    ((2, 3, 384, 128), False, torch.float16, 0),
    ((2, 3, 384, 128), True, torch.bfloat16, 4),
    ((1, 5, 300, 64), True, torch.float16, 1),
    ((1, 2, 257, 64), False, torch.bfloat16, 64),   # more chunks than slices, ragged S
])
def test_bwd_host_entry_matches_device_entry(shape, causal, dtype, chunks):
    """fmha_bwd_host against fmha_bwd on the same inputs.  A key block's dK and
    dV are summed in TMEM in a fixed order, so they are bit-identical.  dQ adds
    the key blocks' fp32 parts in an unspecified order, so the two may differ
    by the rounding of that order: one unit in the last place of the 16-bit
    result, plus fp32 cancellation noise near zero."""
    B, H, S, D = shape
    w = synthetic.Workload("bhost", B, H, S, D, "f16" if dtype == torch.float16 else "bf16",
                           causal, 1.0, 321 + S)
    q, k, v = synthetic.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    d_o = torch.randn(q.shape, generator=g).to(q.dtype)
    o, lse = wsa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale)
    ref = wsa.attention_backward(q.cuda(), k.cuda(), v.cuda(), o, lse, d_o.cuda(), causal=causal,
                                 scale=w.scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    hin = [t.cpu().pin_memory() for t in (q, k, v, o, lse, d_o)]
    hout = [torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory() for _ in range(3)]
    wsa.fmha_bwd_host(*hin, *hout, causal=causal, scale=w.scale, n_chunks=chunks)
    assert wsa.get_device_status() == wsa.FMHA_OK
    dq_h, dk_h, dv_h = hout
    dq_r, dk_r, dv_r = (t.cpu() for t in ref)
    assert torch.equal(dk_h, dk_r) and torch.equal(dv_h, dv_r)
    ulp = 2.0 ** -10 if dtype == torch.float16 else 2.0 ** -7
    diff = (dq_h.float() - dq_r.float()).abs()
    lim = ulp * dq_r.float().abs() + 1e-5 * float(dq_r.float().abs().max())
    assert bool((diff <= lim).all()), "dQ differs by %.3e" % float(diff.max())


def test_host_entry_e4m3_matches_device_entry():
    """The host-buffer entry with E4M3 inputs (V transposed per head, O bf16):
    bit-identical to fmha_fwd on the same staged tensors."""
    w = synthetic.Workload("host-e4m3", 2, 3, 512, 128, "e4m3", True, 1.0, 88)
    q, k, v = synthetic.make_inputs(w)
    vt = synthetic.kernel_v(v)
    hq, hk, hv = (t.pin_memory() for t in (q, k, vt))
    ho = torch.full(q.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    hl = torch.full(q.shape[:3], float("nan"), dtype=torch.float32).pin_memory()
    q_dev, k_dev, v_dev = (torch.empty_like(t, device="cuda") for t in (q, k, vt))
    o_dev = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse_dev = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    wsa.fmha_fwd_host(hq, hk, hv, ho, hl, q_dev, k_dev, v_dev, o_dev, lse_dev, causal=True,
                      scale=w.scale, n_chunks=3)
    assert wsa.get_device_status() == wsa.FMHA_OK
    o_ref, l_ref = wsa.attention(q.cuda(), k.cuda(), vt.cuda(), causal=True, scale=w.scale)
    assert wsa.get_device_status() == wsa.FMHA_OK
    assert torch.equal(ho, o_ref.cpu()) and torch.equal(hl, l_ref.cpu())
