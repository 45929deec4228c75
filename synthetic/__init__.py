"""Seeded synthetic inputs for the attention forward pass.

This module only draws numbers and names shapes.  It holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can consume its
tensors without sharing any of the method's code.

The workload table mirrors the pages' attention benchmark: fp16, batch 4,
32 heads, head dim 128, sequence lengths from 1K to 16K ("Optimal Software
Pipelining and Warp Specialization for Tensor Core GPUs", results section 6.2,
Figs. 7-8 and the claims table; "Tawa", Section V-D).  The pages run on no
public dataset, so seeded i.i.d. N(0,1) draws stand in for activations.

Recipe (one generator per workload):
  * ``torch.Generator('cpu').manual_seed(seed)``, seed = 1000 + workload index;
  * Q, then K, then V drawn with ``torch.randn(B, H, S, D, float32)`` from that
    generator, in that order, then cast (round-to-nearest) to the storage dtype;
  * ``k_mult`` (a power of two) multiplies K after the cast, which is exact; it
    sharpens the softmax for the numerics-stress workload.
Layout is contiguous (B, H, S, D); LSE is (B, H, S) float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str          # "f16", "bf16" or "e4m3" (E4M3 Q, K, V; O in bf16)
    causal: bool
    k_mult: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        # the float32 value 1/sqrt(D), the softmax scale both sides receive
        return float(torch.tensor(1.0 / math.sqrt(self.D), dtype=torch.float32).item())

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f16": torch.float16, "bf16": torch.bfloat16,
                "e4m3": torch.float8_e4m3fn}[self.dtype]

    @property
    def flops(self) -> float:
        """Attention forward flop count 4*B*H*S^2*D, halved under a causal mask."""
        f = 4.0 * self.B * self.H * self.S * self.S * self.D
        return f / 2.0 if self.causal else f

    def describe(self) -> str:
        return ("B%d H%d S%d D%d %s %s%s" % (
            self.B, self.H, self.S, self.D, self.dtype,
            "causal" if self.causal else "non-causal",
            (" K*%g" % self.k_mult) if self.k_mult != 1.0 else ""))


WORKLOADS = [
    Workload("tiny_b1h2s256d64_f16", 1, 2, 256, 64, "f16", False, 1.0, 1000),
    Workload("b4h32s1k_d128_f16", 4, 32, 1024, 128, "f16", False, 1.0, 1001),
    Workload("b4h32s4k_d128_bf16_causal", 4, 32, 4096, 128, "bf16", True, 1.0, 1002),
    Workload("b2h16s8k_d64_f16_causal_ksharp", 2, 16, 8192, 64, "f16", True, 4.0, 1003),
    Workload("b4h32s16k_d128_f16", 4, 32, 16384, 128, "f16", False, 1.0, 1004),
]
HEADLINE = WORKLOADS[4]

# The headline shape with E4M3 inputs: a benchmark and parity line for the
# 8-bit path, not one of the five contract configurations above.
FP8_WORKLOADS = [
    Workload("b4h32s16k_d128_e4m3", 4, 32, 16384, 128, "e4m3", False, 1.0, 1104),
]


def by_name(name: str) -> Workload:
    for w in WORKLOADS + FP8_WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def _scale(t: torch.Tensor, f: float) -> torch.Tensor:
    """t * f in t's dtype (exact for the power-of-two factors used here);
    float8 has no arithmetic of its own, so it goes through float32."""
    if t.dtype == torch.float8_e4m3fn:
        return (t.float() * f).to(t.dtype)
    return t * f


def make_inputs(w: Workload, B=None, H=None, S=None, D=None, dtype=None, seed=None):
    """Seeded (q, k, v) on the CPU, contiguous (B, H, S, D) in the storage dtype.

    Shape/dtype/seed overrides give the small and ragged cases with the same
    recipe as the named workload.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    S = w.S if S is None else S
    D = w.D if D is None else D
    dt = w.torch_dtype if dtype is None else dtype
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    q = torch.randn(B, H, S, D, generator=g, dtype=torch.float32).to(dt)
    k = torch.randn(B, H, S, D, generator=g, dtype=torch.float32).to(dt)
    v = torch.randn(B, H, S, D, generator=g, dtype=torch.float32).to(dt)
    if w.k_mult != 1.0:
        k = _scale(k, w.k_mult)
    return q.contiguous(), k.contiguous(), v.contiguous()


def make_inputs_device(w: Workload, device, seed=None):
    """Same distribution drawn directly on a CUDA device (for timing runs only:
    the values differ from the CPU draw, so parity checks use make_inputs)."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    shape = (w.B, w.H, w.S, w.D)
    out = []
    for _ in range(3):
        out.append(torch.randn(shape, generator=g, device=device,
                               dtype=torch.float32).to(w.torch_dtype))
    q, k, v = out
    if w.k_mult != 1.0:
        k = _scale(k, w.k_mult)
    return q, k, v


def kernel_v(v: torch.Tensor) -> torch.Tensor:
    """V in the layout the kernel takes for its dtype: (B, H, S, D) for 16-bit
    inputs, transposed to (B, H, D, S) for E4M3."""
    if v.dtype == torch.float8_e4m3fn:
        return v.transpose(-1, -2).contiguous()
    return v
