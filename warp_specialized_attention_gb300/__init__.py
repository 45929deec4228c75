"""GB300 (sm_103a) fused attention: the forward O = softmax(scale * Q K^T
[+ causal mask]) V with the per-row natural log-sum-exp, as the three-stage
T/C/U loop of "Tawa: Automatic Warp Specialization for Modern GPUs with
Asynchronous References", Section III-D, Algorithm 1; and its backward pass
(dQ, dK, dV from the forward's O and LSE), on one GPU.

This module is a thin ctypes binding of ``libwsattn.so`` (include/wsattn.h):
it only checks tensor metadata and marshals pointers, sizes and the stream.
Every step of the computation runs in the library's CUDA kernel; there is no
fallback.  If the library has not been built, importing this module succeeds
but every call raises ``LibraryNotBuilt`` -- run
``python -m warp_specialized_attention_gb300.build``.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = [
    "FMHA_OK", "FMHA_ERR_INVALID_ARG", "FMHA_ERR_UNSUPPORTED", "FMHA_ERR_CUDA",
    "FMHA_ERR_TIMEOUT", "FMHA_F16", "FMHA_BF16", "FMHA_E4M3", "FmhaError", "LibraryNotBuilt",
    "library_path", "load_library", "fmha_fwd", "fmha_fwd_host", "fmha_fwd_testing",
    "fmha_fwd_split_testing", "attention",
    "fmha_bwd", "fmha_bwd_workspace_bytes", "fmha_bwd_noalloc", "fmha_bwd_host",
    "fmha_bwd_host_scratch_bytes", "attention_backward", "AttentionFunction",
    "flash_attention",
    "get_device_status", "status_str", "version",
]

FMHA_OK, FMHA_ERR_INVALID_ARG, FMHA_ERR_UNSUPPORTED, FMHA_ERR_CUDA, FMHA_ERR_TIMEOUT = range(5)
FMHA_F16, FMHA_BF16, FMHA_E4M3 = 0, 1, 2

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libwsattn.so")
_lib = None
_lock = threading.Lock()


class LibraryNotBuilt(RuntimeError):
    pass


class FmhaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = "%s: %s" % (where, status_str(status))
        if detail:
            msg += " (%s)" % detail
        super().__init__(msg)


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libwsattn.so (once).  Raises LibraryNotBuilt if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise LibraryNotBuilt(
                "libwsattn.so not found at %s; build it with "
                "`python -m warp_specialized_attention_gb300.build`" % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        fwd_args = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float,
                    ctypes.c_int, vp]
        lib.fmha_fwd.argtypes = fwd_args
        lib.fmha_fwd.restype = ctypes.c_int
        lib.fmha_fwd_host.argtypes = [vp] * 10 + [i64, i64, i64, i64, ctypes.c_int,
                                                  ctypes.c_float, ctypes.c_int, ctypes.c_int, vp]
        lib.fmha_fwd_host.restype = ctypes.c_int
        lib.fmha_fwd_testing.argtypes = fwd_args + [ctypes.c_int, ctypes.c_double, ctypes.c_float]
        lib.fmha_fwd_testing.restype = ctypes.c_int
        lib.fmha_fwd_split_testing.argtypes = fwd_args + [i64]
        lib.fmha_fwd_split_testing.restype = ctypes.c_int
        lib.fmha_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64]
        lib.fmha_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fmha_bwd.argtypes = [vp] * 10 + [ctypes.c_size_t, i64, i64, i64, i64, ctypes.c_int,
                                             ctypes.c_float, ctypes.c_int, vp]
        lib.fmha_bwd.restype = ctypes.c_int
        lib.fmha_bwd_noalloc.argtypes = [vp] * 9 + [i64, i64, i64, i64, ctypes.c_int,
                                                    ctypes.c_float, ctypes.c_int, vp]
        lib.fmha_bwd_noalloc.restype = ctypes.c_int
        lib.fmha_bwd_host_scratch_bytes.argtypes = [i64, i64, i64, i64]
        lib.fmha_bwd_host_scratch_bytes.restype = ctypes.c_size_t
        lib.fmha_bwd_host.argtypes = [vp] * 10 + [ctypes.c_size_t, i64, i64, i64, i64,
                                                  ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                                  ctypes.c_int, vp]
        lib.fmha_bwd_host.restype = ctypes.c_int
        lib.fmha_get_device_status.argtypes = [vp]
        lib.fmha_get_device_status.restype = ctypes.c_int
        lib.fmha_status_str.argtypes = [ctypes.c_int]
        lib.fmha_status_str.restype = ctypes.c_char_p
        lib.fmha_last_cuda_error.argtypes = []
        lib.fmha_last_cuda_error.restype = ctypes.c_char_p
        lib.fmha_version.argtypes = []
        lib.fmha_version.restype = ctypes.c_int
        _lib = lib
        return lib


def status_str(status: int) -> str:
    try:
        return load_library().fmha_status_str(int(status)).decode()
    except LibraryNotBuilt:
        return "status %d" % status


def version() -> int:
    return int(load_library().fmha_version())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FMHA_F16
    if t.dtype == torch.bfloat16:
        return FMHA_BF16
    if t.dtype == torch.float8_e4m3fn:
        return FMHA_E4M3
    raise TypeError("q/k/v must be float16, bfloat16 or float8_e4m3fn, got %s" % t.dtype)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return int(stream.cuda_stream)
    return int(stream)


def _check(q, k, v, o, lse):
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % name)
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    fp8 = q.dtype == torch.float8_e4m3fn
    if q.dim() != 4 or q.shape != k.shape or q.shape != o.shape:
        raise ValueError("q, k, o must share one (B, H, S, D) shape")
    B, H, S, D = q.shape
    if tuple(v.shape) != ((B, H, D, S) if fp8 else (B, H, S, D)):
        raise ValueError("v must be (B, H, S, D), or (B, H, D, S) (transposed) for float8_e4m3fn")
    if not (q.dtype == k.dtype == v.dtype) or o.dtype != (torch.bfloat16 if fp8 else q.dtype):
        raise TypeError("q, k, v must share one dtype; o has it too, or is bfloat16 for "
                        "float8_e4m3fn inputs")
    if lse.dtype != torch.float32 or tuple(lse.shape) != tuple(q.shape[:3]):
        raise ValueError("lse must be float32 of shape (B, H, S)")
    devs = {t.device for t in (q, k, v, o, lse)}
    if len(devs) != 1:
        raise ValueError("all tensors must be on one device")


def fmha_fwd(q, k, v, o, lse, causal: bool = False, scale: float | None = None,
             stream=None) -> None:
    """Enqueue the forward kernel: o, lse <- attention(q, k, v).

    q, k, v, o: contiguous (B, H, S, D) CUDA tensors of one dtype (f16/bf16);
    or q, k float8_e4m3fn (B, H, S, D), v float8_e4m3fn transposed (B, H, D, S)
    and o bfloat16 (B, H, S, D).  lse: contiguous (B, H, S) float32.  scale
    defaults to the float32 value of 1/sqrt(D).  Asynchronous on ``stream``
    (default: torch's current stream).
    """
    lib = load_library()
    _check(q, k, v, o, lse)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        st = lib.fmha_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr(), B, H, S, D, int(bool(causal)), float(scale),
                          _dtype_code(q), _stream_handle(stream))
    if st != FMHA_OK:
        raise FmhaError(st, "fmha_fwd", lib.fmha_last_cuda_error().decode())


def fmha_fwd_host(q, k, v, o, lse, q_dev, k_dev, v_dev, o_dev, lse_dev, causal: bool = False,
                  scale: float | None = None, n_chunks: int = 0, stream=None) -> None:
    """Enqueue attention on host tensors with overlapped transfers (C ABI
    fmha_fwd_host): q, k, v, o (B, H, S, D) and lse (B, H, S) float32 are CPU
    tensors (pinned for overlap); q_dev, k_dev, v_dev, o_dev, lse_dev are CUDA
    staging tensors of the same shapes and dtypes.  Synchronise ``stream``
    before reading o, lse.
    """
    lib = load_library()
    _check(q_dev, k_dev, v_dev, o_dev, lse_dev)
    for name, t, d in (("q", q, q_dev), ("k", k, k_dev), ("v", v, v_dev), ("o", o, o_dev),
                       ("lse", lse, lse_dev)):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise ValueError("%s must be a CPU tensor" % name)
        if not t.is_contiguous() or t.shape != d.shape or t.dtype != d.dtype:
            raise ValueError("%s must be contiguous and match its staging tensor" % name)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q_dev.device):
        st = lib.fmha_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), q_dev.data_ptr(), k_dev.data_ptr(),
                               v_dev.data_ptr(), o_dev.data_ptr(), lse_dev.data_ptr(), B, H, S, D,
                               int(bool(causal)), float(scale), _dtype_code(q), int(n_chunks),
                               _stream_handle(stream))
    if st != FMHA_OK:
        raise FmhaError(st, "fmha_fwd_host", lib.fmha_last_cuda_error().decode())


def fmha_fwd_testing(q, k, v, o, lse, causal: bool, scale: float, inject_fault: int,
                     wait_limit_s: float, tau: float = 15.0, stream=None) -> int:
    """Test hook of include/wsattn_testing.h; returns the raw status code."""
    lib = load_library()
    _check(q, k, v, o, lse)
    B, H, S, D = q.shape
    with torch.cuda.device(q.device):
        return int(lib.fmha_fwd_testing(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), B, H, S, D, int(bool(causal)),
                                        float(scale), _dtype_code(q), _stream_handle(stream),
                                        int(inject_fault), float(wait_limit_s), float(tau)))


def fmha_fwd_split_testing(q, k, v, o, lse, causal: bool, scale: float, split_units: int,
                           stream=None) -> int:
    """Test hook of include/wsattn_testing.h (the number of key-split units
    of the last wave); returns the raw status code."""
    lib = load_library()
    _check(q, k, v, o, lse)
    B, H, S, D = q.shape
    with torch.cuda.device(q.device):
        return int(lib.fmha_fwd_split_testing(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                              o.data_ptr(), lse.data_ptr(), B, H, S, D,
                                              int(bool(causal)), float(scale), _dtype_code(q),
                                              _stream_handle(stream), int(split_units)))


def get_device_status(stream=None, device=None) -> int:
    """Synchronise the stream; return (and clear) the device status code."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        return int(lib.fmha_get_device_status(_stream_handle(stream)))


def attention(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocate O (dtype of q; bfloat16 for float8_e4m3fn inputs) and LSE
    (float32) with torch and run fmha_fwd.  For float8_e4m3fn, v is given
    transposed, (B, H, D, S)."""
    o = torch.empty(q.shape, device=q.device,
                    dtype=torch.bfloat16 if q.dtype == torch.float8_e4m3fn else q.dtype)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fmha_fwd(q, k, v, o, lse, causal=causal, scale=scale, stream=stream)
    return o, lse


def fmha_bwd_workspace_bytes(B: int, H: int, S: int, D: int) -> int:
    """Bytes of device scratch fmha_bwd needs (C ABI fmha_bwd_workspace_bytes)."""
    return int(load_library().fmha_bwd_workspace_bytes(B, H, S, D))


def fmha_bwd(q, k, v, o, lse, d_o, dq, dk, dv, workspace=None, causal: bool = False,
             scale: float | None = None, stream=None) -> None:
    """Enqueue the backward pass (C ABI fmha_bwd): dq, dk, dv <- gradients of
    attention(q, k, v) for the output gradient d_o, using the forward's o and
    lse.  All (B, H, S, D) 16-bit CUDA tensors of one dtype, lse float32
    (B, H, S).  ``workspace`` is a CUDA uint8 tensor of at least
    fmha_bwd_workspace_bytes(B, H, S, D) bytes; one is allocated with torch
    when it is None."""
    lib = load_library()
    _check(q, k, v, o, lse)
    for name, t in (("d_o", d_o), ("dq", dq), ("dk", dk), ("dv", dv)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("%s must match q's shape and dtype" % name)
    B, H, S, D = q.shape
    need = fmha_bwd_workspace_bytes(B, H, S, D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError("workspace must be a CUDA tensor of at least %d bytes" % need)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        st = lib.fmha_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          d_o.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          B, H, S, D, int(bool(causal)), float(scale), _dtype_code(q),
                          _stream_handle(stream))
    if st != FMHA_OK:
        raise FmhaError(st, "fmha_bwd", lib.fmha_last_cuda_error().decode())


def fmha_bwd_noalloc(q, k, v, o, lse, d_o, dq, dk, dv, causal: bool = False,
                     scale: float | None = None, stream=None) -> None:
    """fmha_bwd with the library's own static scratch (C ABI fmha_bwd_noalloc):
    no workspace, a size limit, and calls that overlap in time race."""
    lib = load_library()
    _check(q, k, v, o, lse)
    for name, t in (("d_o", d_o), ("dq", dq), ("dk", dk), ("dv", dv)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("%s must match q's shape and dtype" % name)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        st = lib.fmha_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), d_o.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), B, H, S, D, int(bool(causal)), float(scale),
                                  _dtype_code(q), _stream_handle(stream))
    if st != FMHA_OK:
        raise FmhaError(st, "fmha_bwd_noalloc", lib.fmha_last_cuda_error().decode())


def fmha_bwd_host_scratch_bytes(B: int, H: int, S: int, D: int) -> int:
    """Bytes of device scratch fmha_bwd_host needs (C ABI
    fmha_bwd_host_scratch_bytes)."""
    return int(load_library().fmha_bwd_host_scratch_bytes(B, H, S, D))


def fmha_bwd_host(q, k, v, o, lse, d_o, dq, dk, dv, scratch=None, causal: bool = False,
                  scale: float | None = None, n_chunks: int = 0, stream=None,
                  device=None) -> None:
    """Enqueue the backward pass on host tensors with overlapped transfers (C
    ABI fmha_bwd_host): q, k, v, o, d_o (B, H, S, D) 16-bit and lse (B, H, S)
    float32 are CPU inputs, dq, dk, dv CPU outputs of q's shape and dtype
    (pinned for overlap).  ``scratch`` is a CUDA uint8 tensor of at least
    fmha_bwd_host_scratch_bytes(B, H, S, D) bytes; one is allocated with torch
    on ``device`` (default: the current device) when it is None.  Synchronise
    ``stream`` before reading dq, dk, dv."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("d_o", d_o), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CPU tensor" % name)
        if t.dim() != 4 or t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("%s must match q's (B, H, S, D) shape and dtype" % name)
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("fmha_bwd_host takes float16 or bfloat16 tensors")
    B, H, S, D = q.shape
    if (not isinstance(lse, torch.Tensor) or lse.is_cuda or not lse.is_contiguous()
            or lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, S)):
        raise ValueError("lse must be a contiguous CPU float32 tensor of shape (B, H, S)")
    need = fmha_bwd_host_scratch_bytes(B, H, S, D)
    if scratch is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        scratch = torch.empty(need, dtype=torch.uint8, device=dev)
    if not scratch.is_cuda or scratch.numel() * scratch.element_size() < need:
        raise ValueError("scratch must be a CUDA tensor of at least %d bytes" % need)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(scratch.device):
        st = lib.fmha_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), d_o.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), scratch.data_ptr(),
                               scratch.numel() * scratch.element_size(), B, H, S, D,
                               int(bool(causal)), float(scale), _dtype_code(q), int(n_chunks),
                               _stream_handle(stream))
    if st != FMHA_OK:
        raise FmhaError(st, "fmha_bwd_host", lib.fmha_last_cuda_error().decode())


def attention_backward(q, k, v, o, lse, d_o, causal: bool = False, scale: float | None = None,
                       stream=None):
    """Allocate dq, dk, dv (and the workspace) with torch and run fmha_bwd."""
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fmha_bwd(q, k, v, o, lse, d_o, dq, dk, dv, causal=causal, scale=scale, stream=stream)
    return dq, dk, dv


class AttentionFunction(torch.autograd.Function):
    """Differentiable attention on the library's kernels: the forward runs
    fmha_fwd and keeps O and LSE, the backward runs fmha_bwd with them.
    16-bit (float16 / bfloat16) tensors of shape (B, H, S, D), D 64 or 128;
    E4M3 inputs are forward-only.  LSE is returned as a non-differentiable
    output: a loss that depends on it fails in the forward's autograd graph
    (no gradient flows through it), not at backward time."""

    @staticmethod
    def forward(ctx, q, k, v, causal=False, scale=None):
        if scale is None:
            scale = 1.0 / math.sqrt(q.shape[-1])
        o, lse = attention(q, k, v, causal=causal, scale=scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = bool(causal), float(scale)
        ctx.mark_non_differentiable(lse)
        ctx.set_materialize_grads(False)
        return o, lse

    @staticmethod
    def backward(ctx, d_o, d_lse):
        if d_o is None:   # O does not reach the loss: no gradient for q, k, v
            return None, None, None, None, None
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = attention_backward(q, k, v, o, lse, d_o.contiguous(), causal=ctx.causal,
                                        scale=ctx.scale)
        return dq, dk, dv, None, None


def flash_attention(q, k, v, causal: bool = False, scale: float | None = None):
    """O = softmax(scale * Q K^T [+ causal mask]) V, differentiable with respect
    to q, k and v (AttentionFunction); returns O only."""
    o, _ = AttentionFunction.apply(q, k, v, causal, scale)
    return o
