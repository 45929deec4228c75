"""Benchmark of the fused attention forward on GB300: prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one fmha_fwd over the whole workload (default: B=4, H=32, S=16384,
D=128, fp16, no mask -- the pages' headline attention shape).  The metric is
attention-forward TFLOPS, 4*B*H*S^2*D per step (halved under a causal mask).

ours (default):
  value     K steps with inputs resident in HBM, CUDA events on the launching
            stream, barrier + synchronize on both sides, max over ranks.  The
            inputs (2.15 GB) exceed the 129 MB L2, so no flush between steps.
  e2e       the same metric through the public API with host buffers
            (fmha_fwd_host): per step the pinned-host -> device copy of Q, K, V,
            the kernels and the device -> pinned-host copy of O and LSE, all
            inside the timed region, copies of one chunk of slices overlapped
            with the computation of another.
  roofline  the attention kernel against the measured dense 16-bit tensor peak.
  cpu_baseline  the fp64 CPU oracle on a bounded row sample of the same
            workload on this host's cores (rank 0, N=1 only).
reference:  the fp64 CPU oracle itself, timed the same way on bounded samples.

--pass bwd times the backward pass (fmha_bwd) instead: a step is one backward
over the workload given the forward's O and LSE, counted as 2.5x the forward
FLOPs (five products of 2*S^2*D per head instead of two); its e2e leg copies
Q, K, V, O, LSE, dO in from pinned host memory and dQ, dK, dV out per step,
and its CPU baseline is the fp64 backward oracle on one (batch, head) slice.

Under torchrun (N > 1) every rank runs its own copy of the workload (the
(batch, head) units are independent, so per-GPU work is fixed: weak scaling);
there is no data-path collective, only a barrier and a max of the timings.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

METRIC = "FMHA fwd TFLOPS at B4 H32 S16K D128 fp16; % of GB300 dense tensor peak"
UNIT = "TFLOPS"
KERNEL_SOURCES = ["ptx.cuh", "fmha_fwd_sm103.cuh", "fmha_fwd_d64.cu", "fmha_fwd_d128.cu",
                  "fmha_fwd_e4m3.cu", "fmha_api.cu"]
BWD_SOURCES = ["fmha_bwd_sm103.cuh", "fmha_bwd.cu"]


# ----------------------------------------------------------------------------- helpers

def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def _barrier(dist, device):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def _max_over_ranks(dist, x, device):
    """The slowest rank's time: every rank waits for it (weak scaling)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(w, rank):
    """Each rank draws its own copy of the workload (its own batch): the
    (batch, head) slices are independent, so ranks share no data."""
    return w.seed + 7919 * rank


def job_tflops(w, world, ms_per_step):
    """Whole-job throughput: every rank processed one full workload per step."""
    return world * w.flops / (ms_per_step / 1e3) / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


def _code_only(text):
    """C/C++/CUDA source without comments and blank lines: a comment edit does
    not change the compiled kernel, so it keeps its recorded counters."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def _kernel_sha(sources=None):
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, "warp_specialized_attention_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic(workload_name, sources=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload_name)
    if not e or e.get("kernel_sha") != _kernel_sha(sources):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.path = None
        smi = shutil.which("nvidia-smi")
        if smi is None or device is None:
            return
        ident = str(device.index)
        try:
            uuid = torch.cuda.get_device_properties(device).uuid
            ident = "GPU-" + str(uuid)
        except Exception:
            pass
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.out = open(self.path, "w")
        try:
            self.proc = subprocess.Popen(
                [smi, "-i", ident, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle

def _row_flops(S, D, causal, rows):
    if causal:
        return float(sum(4.0 * (int(i) + 1) * D for i in rows))
    return 4.0 * S * D * len(rows)


class OracleSampler:
    """Bounded samples of the workload for the fp64 CPU oracle: whole rows of
    one (batch, head) slice at a time, rows spread over the sequence."""

    def __init__(self, w, k_head, v_head, q_head):
        import oracle
        self.oracle = oracle
        self.w = w
        self.k = k_head
        self.v = v_head
        self.q = q_head
        self.rng = np.random.default_rng(w.seed)

    def rows(self, n):
        return np.sort(self.rng.choice(self.w.S, size=min(n, self.w.S), replace=False))

    def run(self, rows):
        t0 = time.perf_counter()
        self.oracle.attention_rows(self.q[rows], self.k, self.v, rows, self.w.causal,
                                   self.w.scale)
        dt = time.perf_counter() - t0
        return dt, _row_flops(self.w.S, self.w.D, self.w.causal, rows)

    def rows_for(self, seconds):
        """Calibrate: how many rows take about `seconds` on this host."""
        n = 32
        dt, _ = self.run(self.rows(n))
        while dt < 0.5 and n < self.w.S:
            n = min(self.w.S, n * 4)
            dt, _ = self.run(self.rows(n))
        return max(1, min(self.w.S, int(n * seconds / max(dt, 1e-6))))


def _head_inputs(w, q, k, v, bh):
    """One (batch, head) slice as float64 numpy (exact upcast of the stored values)."""
    b, h = divmod(bh, w.H)
    to = lambda t: t[b, h].double().cpu().numpy()  # noqa: E731
    return to(q), to(k), to(v)


def cpu_baseline(w, q, k, v, seconds=12.0):
    """The oracle on whole (batch, head) slices -- all rows, every visible key --
    until about `seconds` of host time, or on a row sample of one slice when
    one slice alone takes longer."""
    import oracle
    qh, kh, vh = _head_inputs(w, q, k, v, 0)
    smp = OracleSampler(w, kh, vh, qh)
    n = smp.rows_for(seconds)
    if n < w.S:
        rows = smp.rows(n)
        dt, fl = smp.run(rows)
        sample = ("%d query rows (whole rows, every visible key) of one (batch, head) slice "
                  "of %s" % (n, w.describe()))
    else:
        dt = fl = 0.0
        heads = 0
        all_rows = np.arange(w.S)
        while dt < seconds and heads < w.B * w.H:
            qh, kh, vh = _head_inputs(w, q, k, v, heads)
            smp = OracleSampler(w, kh, vh, qh)
            t, f = smp.run(all_rows)
            dt, fl, heads = dt + t, fl + f, heads + 1
        sample = "%d whole (batch, head) slices of %s" % (heads, w.describe())
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": "%s; %.3g GFLOP in %.2f s" % (sample, fl / 1e9, dt)}


# ----------------------------------------------------------------------------- arms

def run_reference(args, w):
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    q, k, v = synthetic.make_inputs(w, B=1, H=1)   # one head: the oracle samples rows of it
    qh, kh, vh = (t[0, 0].double().numpy() for t in (q, k, v))
    smp = OracleSampler(w, kh, vh, qh)
    budget = 150.0  # whole run, seconds
    per_step = max(0.5, min(6.0, budget / max(1, args.steps + args.warmup)))
    n = smp.rows_for(per_step)
    for _ in range(args.warmup):
        smp.run(smp.rows(n))
    total_t = total_f = 0.0
    for _ in range(args.steps):
        dt, fl = smp.run(smp.rows(n))
        total_t += dt
        total_f += fl
    value = total_f / total_t / 1e12
    sample = ("each step: %d query rows (whole rows) of one (batch, head) slice of %s"
              % (n, w.describe()))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129 * 10 ** 6  # GB300 L2


def _config(w, in_bytes=None, flushed=None):
    """The workload, and how the timed steps treat L2: inputs larger than L2
    run back to back; inputs that fit are evicted between timed launches."""
    if in_bytes is None:
        in_bytes = 3 * w.B * w.H * w.S * w.D * (1 if w.dtype == "e4m3" else 2)
    if flushed is None:
        l2 = "inputs %.3f GB (timed on the host cores: no GPU L2)" % (in_bytes / 1e9)
    elif flushed:
        l2 = ("inputs %.3f GB fit in the 129 MB L2: %d MB written between timed launches, "
              "outside their events" % (in_bytes / 1e9, 2 * L2_BYTES // 10 ** 6))
    else:
        l2 = "inputs %.2f GB > 129 MB L2: no flush between steps" % (in_bytes / 1e9)
    return {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "dtype": w.dtype,
            "causal": w.causal, "k_mult": w.k_mult, "scale": w.scale,
            "layout": "BHSD contiguous, LSE fp32 (B,H,S)", "l2": l2}


def _timed_steps(step, n, stream, device, in_bytes):
    """n calls of step() on `stream`, one CUDA event pair per call.  Inputs
    larger than L2 run back to back and the total is first to last event.
    Inputs that fit in L2 are evicted before every call by writing twice the
    L2 size, outside the call's own events, and the total is the sum of the
    calls' times.  Returns (per-call ms, total ms, whether L2 was flushed)."""
    flush = (torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
             if in_bytes <= L2_BYTES else None)
    if flush is None:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        ev[0].record(stream)
        for i in range(n):
            step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(device)
        launches = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
        return launches, ev[0].elapsed_time(ev[-1]), False
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        with torch.cuda.stream(stream):
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    launches = [starts[i].elapsed_time(ends[i]) for i in range(n)]
    return launches, sum(launches), True


def run_ours(args, w):
    import warp_specialized_attention_gb300 as wsa
    world, rank, local = _dist_env()
    dist = _init_dist(world)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the attention path has no CPU fallback)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wsa.load_library()

    q, k, v_rows = synthetic.make_inputs_device(w, device, seed=rank_seed(w, rank))
    fp8 = w.dtype == "e4m3"
    v = synthetic.kernel_v(v_rows)           # E4M3 V goes in transposed, (B, H, D, S)
    o = torch.empty(q.shape, device=device, dtype=torch.bfloat16 if fp8 else q.dtype)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    for _ in range(args.warmup):
        wsa.fmha_fwd(q, k, v, o, lse, causal=w.causal, scale=w.scale, stream=stream)
    torch.cuda.synchronize(device)
    if wsa.get_device_status(stream) != wsa.FMHA_OK:
        raise SystemExit("device status error after warm-up")

    # ---- device-resident timing: one event pair per launch, on the launch stream
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    sampler = ClockSampler(device) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    _barrier(dist, device)
    torch.cuda.synchronize(device)
    launches, total_ms, flushed = _timed_steps(
        lambda: wsa.fmha_fwd(q, k, v, o, lse, causal=w.causal, scale=w.scale, stream=stream),
        args.steps, stream, device, in_bytes)
    _barrier(dist, device)
    clocks = sampler.stop() if sampler else None
    total_ms = _max_over_ranks(dist, total_ms, device)
    if wsa.get_device_status(stream) != wsa.FMHA_OK:
        raise SystemExit("device status error in the timed region")

    ms_per_step = total_ms / args.steps
    value = job_tflops(w, world, ms_per_step)
    kernel_ms = statistics.mean(launches)
    achieved = w.flops / (kernel_ms / 1e3) / 1e12

    # ---- end to end through the public API with pinned host buffers: every
    # step copies Q, K, V in and O, LSE out (fmha_fwd_host overlaps the copies of
    # one chunk of (batch, head) slices with the computation of the next).
    e2e_steps = max(3, min(args.steps, 20))
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    def e2e_step():
        wsa.fmha_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, o, lse, causal=w.causal,
                          scale=w.scale, n_chunks=args.chunks, stream=stream)

    e2e_step()
    torch.cuda.synchronize(device)
    _barrier(dist, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = _max_over_ranks(dist, e0.elapsed_time(e1), device) / e2e_steps
    e2e_value = job_tflops(w, world, e2e_ms)
    # a step's result really is back on the host
    if not (torch.isfinite(hl).all().item() and torch.isfinite(ho[0, 0, :4].float()).all().item()):
        raise SystemExit("end-to-end outputs are not finite")

    peaks, peak_src = _peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))  # fp16 dense peak equals bf16's
    peak_note = "%s bf16 burst dense (fp16 nominal ratio 1)" % peak_src
    if fp8:   # dense E4M3 runs at twice the 16-bit rate (4.5 vs 2.25 PFLOP/s nominal)
        peak *= 2
        peak_note = "%s bf16 burst dense x 2 (nominal e4m3/bf16 ratio)" % peak_src
    traffic = _traffic(w.name)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q, k, v_rows)

    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic", "config": _config(w, in_bytes, flushed),
        "frac_of_peak": value / world / peak,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d * world,
                "d2h_bytes_per_step": d2h * world, "ms_per_step": e2e_ms,
                "api": "fmha_fwd_host, pinned host buffers, %s chunks" % (args.chunks or 16)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_note,
                     "kernel_ms_mean": kernel_ms, "kernel_ms_min": min(launches)},
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_bwd(args, w):
    import oracle
    import warp_specialized_attention_gb300 as wsa
    world, rank, local = _dist_env()
    dist = _init_dist(world)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the attention path has no CPU fallback)")
    if w.dtype == "e4m3":
        raise SystemExit("the backward pass takes 16-bit inputs")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wsa.load_library()
    q, k, v = synthetic.make_inputs_device(w, device, seed=rank_seed(w, rank))
    g = torch.Generator(device=device)
    g.manual_seed(rank_seed(w, rank) + 1)
    d_o = torch.randn(q.shape, generator=g, device=device, dtype=torch.float32).to(q.dtype)
    o, lse = wsa.attention(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(wsa.fmha_bwd_workspace_bytes(w.B, w.H, w.S, w.D), dtype=torch.uint8,
                     device=device)
    stream = torch.cuda.current_stream(device)
    step = lambda: wsa.fmha_bwd(q, k, v, o, lse, d_o, dq, dk, dv, workspace=ws,  # noqa: E731
                                causal=w.causal, scale=w.scale, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    if wsa.get_device_status(stream) != wsa.FMHA_OK:
        raise SystemExit("device status error after warm-up")
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, o, lse, d_o))
    sampler = ClockSampler(device) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    _barrier(dist, device)
    torch.cuda.synchronize(device)
    launches, total_ms, flushed = _timed_steps(step, args.steps, stream, device, in_bytes)
    _barrier(dist, device)
    clocks = sampler.stop() if sampler else None
    total_ms = _max_over_ranks(dist, total_ms, device)
    if wsa.get_device_status(stream) != wsa.FMHA_OK:
        raise SystemExit("device status error in the timed region")
    flops = 2.5 * w.flops
    ms_per_step = total_ms / args.steps
    value = world * flops / (ms_per_step / 1e3) / 1e12
    step_ms = statistics.mean(launches)
    achieved = flops / (step_ms / 1e3) / 1e12

    # e2e: inputs in from pinned host memory, gradients out, every step, through
    # fmha_bwd_host (chunks of (batch, head) slices, copies overlapping the work)
    hin = [t.cpu().pin_memory() for t in (q, k, v, o, lse, d_o)]
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    scratch = torch.empty(wsa.fmha_bwd_host_scratch_bytes(w.B, w.H, w.S, w.D), dtype=torch.uint8,
                          device=device)

    def e2e_step():
        wsa.fmha_bwd_host(*hin, *hout, scratch=scratch, causal=w.causal, scale=w.scale,
                          n_chunks=args.chunks, stream=stream)

    e2e_steps = max(3, min(args.steps, 10))
    e2e_step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = _max_over_ranks(dist, e0.elapsed_time(e1), device) / e2e_steps
    if not all(torch.isfinite(t[0, 0, :4].float()).all().item() for t in hout):
        raise SystemExit("end-to-end gradients are not finite")

    peaks, peak_src = _peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qh, kh, vh, doh = (t[0, 0].double().cpu().numpy() for t in (q, k, v, d_o))
        t0 = time.perf_counter()
        oracle.attention_bwd(qh, kh, vh, doh, w.causal, w.scale)
        dt = time.perf_counter() - t0
        cpu = {"value": 2.5 * w.flops / (w.B * w.H) / dt / 1e12, "unit": UNIT,
               "cores": oracle.threads(), "kind": "oracle",
               "sample": "one whole (batch, head) slice of %s, backward oracle, %.2f s"
                         % (w.describe(), dt)}
    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {
        "metric": "FMHA bwd TFLOPS (2.5x forward FLOPs) at %s" % w.describe(), "value": value,
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(_config(w, in_bytes, flushed), **{"pass": "backward"}),
        "e2e": {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world,
                "ms_per_step": e2e_ms, "api": "fmha_bwd_host, pinned host buffers, %s chunks" % (args.chunks or 16)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": _traffic(w.name + "_bwd", KERNEL_SOURCES + BWD_SOURCES),
                     "peak_source": "%s bf16 burst dense (fp16 nominal ratio 1)" % peak_src,
                     "step_ms_mean": step_ms, "step_ms_min": min(launches),
                     "note": "a step is 4 launches (memset, delta, backward, dQ conversion)"},
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": 3 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synthetic.HEADLINE.name,
                    choices=[x.name for x in synthetic.WORKLOADS + synthetic.FP8_WORKLOADS])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunks", type=int, default=0,
                    help="(batch, head) chunks for the end-to-end leg (0: library default)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (smaller profiling captures)")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward pass")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 untimed warm-up steps
    w = synthetic.by_name(args.workload)
    if args.batch is not None:
        w = dataclasses.replace(w, B=args.batch, name="%s_b%d" % (w.name, args.batch))
    if args.impl == "reference":
        return run_reference(args, w)
    if args.pass_ == "bwd":
        return run_ours_bwd(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
