"""The C ABI from host threads that have made no CUDA call of their own.

A framework may call the library from a worker thread (torch's autograd
engine runs the backward pass on one) on which no CUDA context is current
yet.  Every entry point must bind the device's context itself: the tensor-map
encoder it calls first is a driver-API function that needs one.  Each thread
below makes its first CUDA call through the library, and the results must be
bit-identical to the same calls made on the main thread."""
import threading

import pytest
import torch

import synthetic
import warp_specialized_attention_gb300 as wsa

pytestmark = pytest.mark.gpu


def _in_fresh_thread(fn):
    box = {}

    def run():
        try:
            box["out"] = fn()
        except BaseException as e:  # re-raised on the caller's thread
            box["err"] = e

    t = threading.Thread(target=run)
    t.start()
    t.join(timeout=120)
    assert not t.is_alive()
    if "err" in box:
        raise box["err"]
    return box["out"]


def test_forward_and_backward_from_fresh_threads():
    w = synthetic.Workload("thread", 2, 3, 520, 64, "f16", True, 1.0, 31)
    q, k, v = (t.cuda() for t in synthetic.make_inputs(w))
    d_o = torch.randn(q.shape, generator=torch.Generator().manual_seed(5)).to(q.dtype).cuda()
    o_ref, lse_ref = wsa.attention(q, k, v, causal=True, scale=w.scale)
    grads_ref = wsa.attention_backward(q, k, v, o_ref, lse_ref, d_o, causal=True, scale=w.scale)
    torch.cuda.synchronize()

    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda", dtype=torch.float32)

    def fwd():
        wsa.fmha_fwd(q, k, v, o, lse, causal=True, scale=w.scale)
        return wsa.get_device_status()

    assert _in_fresh_thread(fwd) == wsa.FMHA_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)

    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    ws = torch.empty(wsa.fmha_bwd_workspace_bytes(*q.shape), dtype=torch.uint8, device="cuda")

    def bwd():
        wsa.fmha_bwd(q, k, v, o, lse, d_o, dq, dk, dv, workspace=ws, causal=True, scale=w.scale)
        return wsa.get_device_status()

    assert _in_fresh_thread(bwd) == wsa.FMHA_OK
    assert torch.equal(dk, grads_ref[1]) and torch.equal(dv, grads_ref[2])
    tol = 1e-3 * grads_ref[0].float().abs().max().item()
    assert (dq.float() - grads_ref[0].float()).abs().max().item() <= tol
