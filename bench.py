"""Benchmark of the fused attention forward on GB300: prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--pass fwd|bwd] [--configs all|none]

A step is one fmha_fwd over the whole workload (default: B=4, H=32, S=16384,
D=128, fp16, no mask -- the pages' headline attention shape).  The metric is
attention-forward TFLOPS, 4*B*H*S^2*D per step (halved under a causal mask).

ours (default):
  value     K steps with inputs resident in HBM, CUDA events on the launching
            stream, barrier + synchronize on both sides, max over ranks.  The
            headline inputs (1.61 GB) exceed the 129 MB L2, so no flush between
            steps; a workload whose inputs fit in L2 is flushed before every
            timed launch, outside its events.
  e2e       the same metric through the public API with host buffers
            (fmha_fwd_host): per step the pinned-host -> device copy of Q, K, V,
            the kernels and the device -> pinned-host copy of O and LSE, all
            inside the timed region, copies of one chunk of slices overlapped
            with the computation of another.  Beside it, the host link's own
            H2D / D2H GB/s, measured with plain copies of the same tensors, so
            a change of the end-to-end figure can be told from a change of link.
  roofline  the attention kernel against the measured dense 16-bit tensor peak.
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload
            on this host's cores (rank 0, N=1 only).
  parity    the timed launch's own output compared with what the oracle
            computed for that sample.
  configs   (N=1, default run) the same record for every other named
            workload: the four smaller forward configurations, the E4M3
            forward and the backward pass of the headline shape.
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

# the headline metric, named exactly as the benchmark's reference quotes it
METRIC = "FMHA fwd TFLOPS at B4 H32 S16K D128 fp16; % of GB300 dense tensor peak"
UNIT = "TFLOPS"
KERNEL_SOURCES = ["ptx.cuh", "fmha_fwd_sm103.cuh", "fmha_fwd_d64.cu", "fmha_fwd_d128.cu",
                  "fmha_fwd_e4m3.cu", "fmha_fwd_ksplit.cu", "fmha_api.cu"]
BWD_SOURCES = ["fmha_bwd_sm103.cuh", "fmha_bwd.cu"]
TOL_O, TOL_LSE = 1e-2, 1e-3       # the forward parity bar for 16-bit inputs


def metric_for(w, pass_="fwd"):
    """The metric a line reports: the headline's own name for the headline
    forward, else one that names the workload it was measured on."""
    if pass_ == "bwd":
        return "FMHA bwd TFLOPS (2.5x forward FLOPs) at %s" % w.describe()
    if w.name == synthetic.HEADLINE.name:
        return METRIC
    return "FMHA fwd TFLOPS at %s; %% of GB300 dense tensor peak" % w.describe()


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
        """Returns (seconds, flops, (o, lse)) for the given query rows."""
        t0 = time.perf_counter()
        out = self.oracle.attention_rows(self.q[rows], self.k, self.v, rows, self.w.causal,
                                         self.w.scale)
        dt = time.perf_counter() - t0
        return dt, _row_flops(self.w.S, self.w.D, self.w.causal, rows), out

    def rows_for(self, seconds):
        """Calibrate: how many rows take about `seconds` on this host."""
        n = 32
        dt, _, _ = self.run(self.rows(n))
        while dt < 0.5 and n < self.w.S:
            n = min(self.w.S, n * 4)
            dt, _, _ = self.run(self.rows(n))
        return max(1, min(self.w.S, int(n * seconds / max(dt, 1e-6))))


def _head_inputs(w, q, k, v, bh):
    """One (batch, head) slice as float64 numpy (exact upcast of the stored values)."""
    b, h = divmod(bh, w.H)
    to = lambda t: t[b, h].double().cpu().numpy()  # noqa: E731
    return to(q), to(k), to(v)


def cpu_baseline(w, q, k, v, seconds=12.0):
    """The oracle on whole (batch, head) slices -- all rows, every visible key --
    until about `seconds` of host time, or on a row sample of one slice when
    one slice alone takes longer.  Returns the baseline record and what the
    oracle computed: a list of (bh, rows, o, lse) for the parity check."""
    import oracle
    qh, kh, vh = _head_inputs(w, q, k, v, 0)
    smp = OracleSampler(w, kh, vh, qh)
    n = smp.rows_for(seconds)
    if n < w.S:
        rows = smp.rows(n)
        dt, fl, out = smp.run(rows)
        computed = [(0, rows, out[0], out[1])]
        sample = ("%d query rows (whole rows, every visible key) of one (batch, head) slice "
                  "of %s" % (n, w.describe()))
    else:
        dt = fl = 0.0
        heads = 0
        computed = []
        all_rows = np.arange(w.S)
        # whole slices spread over the (batch, head) range
        order = np.random.default_rng(w.seed + 1).permutation(w.B * w.H)
        while dt < seconds and heads < w.B * w.H:
            bh = int(order[heads])
            qh, kh, vh = _head_inputs(w, q, k, v, bh)
            smp = OracleSampler(w, kh, vh, qh)
            t, f, out = smp.run(all_rows)
            dt, fl, heads = dt + t, fl + f, heads + 1
            computed.append((bh, all_rows, out[0], out[1]))
        sample = "%d whole (batch, head) slices of %s" % (heads, w.describe())
    rec = {"value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
           "sample": "%s; %.3g GFLOP in %.2f s" % (sample, fl / 1e9, dt)}
    return rec, computed


def _e4m3_o_bound(q64, k64, v64, rows, causal, scale, o_ref, lse_ref, tau=8.0):
    """Per-element bound on |O_gpu - O_oracle| for E4M3 inputs: P is rounded to
    E4M3 (relative 2^-4 for normal values, 2^-10 absolute below 2^-6, i.e.
    2^(-18+tau) of the row's largest term), O to bf16 (2^-8), plus 1e-4 for
    fp32 and ex2.  The attention of |V| comes from the oracle."""
    import oracle
    o_abs, _ = oracle.attention_rows(q64, k64, np.abs(v64), rows, causal, scale)
    out = np.empty_like(o_ref)
    key = np.arange(k64.shape[0])
    for c in range(0, len(rows), 512):
        r = rows[c:c + 512]
        s = (q64[c:c + 512] @ k64.T) * scale
        vis = key[None, :] <= r[:, None] if causal else np.ones(s.shape, dtype=bool)
        s_max = np.where(vis, s, -np.inf).max(axis=1)
        inv_l = np.exp(s_max - lse_ref[c:c + 512])[:, None]
        sum_abs_v = vis.astype(np.float64) @ np.abs(v64)
        out[c:c + 512] = (2.0 ** -4 * o_abs[c:c + 512] + 2.0 ** (-18 + tau) * sum_abs_v * inv_l
                          + 2.0 ** -8 * np.abs(o_ref[c:c + 512]) + 1e-4)
    return out


def fwd_parity(w, q, k, v_rows, o, lse, computed):
    """The GPU output of the timed launches against the oracle's values for
    the CPU baseline's sample (same stored inputs, upcast)."""
    worst_o = worst_l = worst_ratio = 0.0
    n_rows = 0
    for bh, rows, o_ref, lse_ref in computed:
        b, h = divmod(bh, w.H)
        idx = torch.as_tensor(rows, device=o.device)
        og = o[b, h].index_select(0, idx).double().cpu().numpy()
        lg = lse[b, h].index_select(0, idx).double().cpu().numpy()
        if not (np.isfinite(og).all() and np.isfinite(lg).all()):
            return {"pass": False, "note": "non-finite output"}
        d_o = np.abs(og - o_ref)
        worst_o = max(worst_o, float(d_o.max()))
        worst_l = max(worst_l, float(np.abs(lg - lse_ref).max()))
        n_rows += len(rows)
        if w.dtype == "e4m3":
            q64, k64, v64 = (t[b, h].double().cpu().numpy() for t in (q, k, v_rows))
            bound = _e4m3_o_bound(q64[rows], k64, v64, rows, w.causal, w.scale, o_ref, lse_ref)
            worst_ratio = max(worst_ratio, float((d_o / bound).max()))
    rec = {"rows": n_rows, "slices": len(computed), "max_err_o": worst_o,
           "max_err_lse": worst_l, "tol_lse": TOL_LSE}
    if w.dtype == "e4m3":
        rec["o_err_over_e4m3_bound"] = worst_ratio
        rec["tol_o"] = "per element: 2^-4 A(|V|) + 2^-10 sum|v|/l + 2^-8 |O| + 1e-4"
        rec["pass"] = worst_ratio <= 1.0 and worst_l <= TOL_LSE
    else:
        rec["tol_o"] = TOL_O
        rec["pass"] = worst_o <= TOL_O and worst_l <= TOL_LSE
    return rec


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
        dt, fl, _ = smp.run(smp.rows(n))
        total_t += dt
        total_f += fl
    value = total_f / total_t / 1e12
    sample = ("each step: %d query rows (whole rows) of one (batch, head) slice of %s"
              % (n, w.describe()))
    line = {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": UNIT,
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
# Spin before each timed launch of an L2-sized workload, after the flush: the
# host enqueues the launch (ctypes, checks, three tensor-map encodings) while
# the GPU spins, so the launch's start event never waits on the host.
HOST_HEADROOM_CYCLES = 400_000   # ~0.2 ms at 2 GHz


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
            torch.cuda._sleep(HOST_HEADROOM_CYCLES)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    launches = [starts[i].elapsed_time(ends[i]) for i in range(n)]
    return launches, sum(launches), True


def _enqueue_us(step, stream, device, reps=5):
    """Host time to enqueue one step (median of a few), for the record."""
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        step()
        ts.append((time.perf_counter() - t0) * 1e6)
    torch.cuda.synchronize(device)
    return statistics.median(ts)


def _host_link(pairs_in, pairs_out, stream, device, reps=3):
    """GB/s of plain pinned-host <-> device copies of one step's tensors on
    `stream` (all inputs in, then all outputs out, timed apart); best of reps."""
    h2d = sum(h.numel() * h.element_size() for h, _ in pairs_in)
    d2h = sum(h.numel() * h.element_size() for h, _ in pairs_out)
    best_in = best_out = float("inf")
    for _ in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        with torch.cuda.stream(stream):
            e[0].record(stream)
            for h, d in pairs_in:
                d.copy_(h, non_blocking=True)
            e[1].record(stream)
            for h, d in pairs_out:
                h.copy_(d, non_blocking=True)
            e[2].record(stream)
        torch.cuda.synchronize(device)
        best_in = min(best_in, e[0].elapsed_time(e[1]))
        best_out = min(best_out, e[1].elapsed_time(e[2]))
    return h2d / best_in / 1e6, d2h / best_out / 1e6


def _clocks_ok(clocks):
    return clocks is None or not (set(clocks.get("reasons", [])) &
                                  {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"})


def fwd_record(args, w, device, dist, world, rank, cpu_seconds):
    """Measure the forward pass on workload w: one record (the bench line's
    fields), or None on ranks other than 0."""
    import warp_specialized_attention_gb300 as wsa
    q, k, v_rows = synthetic.make_inputs_device(w, device, seed=rank_seed(w, rank))
    fp8 = w.dtype == "e4m3"
    v = synthetic.kernel_v(v_rows)           # E4M3 V goes in transposed, (B, H, D, S)
    o = torch.empty(q.shape, device=device, dtype=torch.bfloat16 if fp8 else q.dtype)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        wsa.fmha_fwd(q, k, v, o, lse, causal=w.causal, scale=w.scale, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    if wsa.get_device_status(stream) != wsa.FMHA_OK:
        raise SystemExit("device status error after warm-up (%s)" % w.name)
    enqueue_us = _enqueue_us(step, stream, device)

    # ---- device-resident timing: one event pair per launch, on the launch stream
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    sampler = ClockSampler(device) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    _barrier(dist, device)
    torch.cuda.synchronize(device)
    launches, total_ms, flushed = _timed_steps(step, args.steps, stream, device, in_bytes)
    _barrier(dist, device)
    clocks = sampler.stop() if sampler else None
    total_ms = _max_over_ranks(dist, total_ms, device)
    if wsa.get_device_status(stream) != wsa.FMHA_OK:
        raise SystemExit("device status error in the timed region (%s)" % w.name)

    ms_per_step = total_ms / args.steps
    value = job_tflops(w, world, ms_per_step)
    kernel_ms = statistics.mean(launches)
    achieved = w.flops / (kernel_ms / 1e3) / 1e12

    # ---- CPU baseline and parity of the timed launches' output (rank 0, N=1)
    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, computed = cpu_baseline(w, q, k, v_rows, seconds=cpu_seconds)
        parity = fwd_parity(w, q, k, v_rows, o, lse, computed)
        parity["sample"] = "the CPU baseline's sample, against the last timed launch's output"

    # ---- end to end through the public API with pinned host buffers: every
    # step copies Q, K, V in and O, LSE out (fmha_fwd_host overlaps the copies of
    # one chunk of (batch, head) slices with the computation of the next).
    e2e_steps = max(3, min(args.steps, 20))
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    q_dev, k_dev, v_dev = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    o_dev, lse_dev = torch.empty_like(o), torch.empty_like(lse)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    h2d_gbs, d2h_gbs = _host_link([(hq, q_dev), (hk, k_dev), (hv, v_dev)],
                                  [(ho, o_dev), (hl, lse_dev)], stream, device)

    def e2e_step():
        wsa.fmha_fwd_host(hq, hk, hv, ho, hl, q_dev, k_dev, v_dev, o_dev, lse_dev,
                          causal=w.causal, scale=w.scale, n_chunks=args.chunks, stream=stream)

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
        raise SystemExit("end-to-end outputs are not finite (%s)" % w.name)

    peaks, peak_src = _peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))  # fp16 dense peak equals bf16's
    peak_note = "%s bf16 burst dense (fp16 nominal ratio 1)" % peak_src
    if fp8:   # dense E4M3 runs at twice the 16-bit rate (4.5 vs 2.25 PFLOP/s nominal)
        peak *= 2
        peak_note = "%s bf16 burst dense x 2 (nominal e4m3/bf16 ratio)" % peak_src
    if rank != 0:
        return None
    return {
        "metric": metric_for(w), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic", "config": _config(w, in_bytes, flushed),
        "frac_of_peak": value / world / peak,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d * world,
                "d2h_bytes_per_step": d2h * world, "ms_per_step": e2e_ms,
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                "link_ms": max(h2d / h2d_gbs, d2h / d2h_gbs) / 1e6,
                "api": "fmha_fwd_host, pinned host buffers, %s chunks" % (args.chunks or 16),
                "link_note": "h2d_gbs / d2h_gbs: plain pinned copies of one step's inputs "
                             "/ outputs on this host link; link_ms: the slower direction's "
                             "time for one step's bytes"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": _traffic(w.name),
                     "peak_source": peak_note,
                     "kernel_ms_mean": kernel_ms, "kernel_ms_min": min(launches),
                     "kernel_ms_median": statistics.median(launches),
                     "host_enqueue_us": enqueue_us},
        "cpu_baseline": cpu,
        "parity": parity,
        "clocks": clocks,
        "clocks_ok": _clocks_ok(clocks),
        "gpu_launches": args.steps,
    }


def bwd_parity(w, got, ref):
    """Backward output of the timed launches (one slice) against the backward
    oracle: per gradient, max |err| <= 1e-2 max|ref| + 1e-3."""
    rec = {"slices": 1, "check": "per gradient: max |err| <= 1e-2 * max|ref| + 1e-3"}
    ok = True
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        err = float(np.abs(g - r).max()) if np.isfinite(g).all() else float("inf")
        lim = 1e-2 * float(np.abs(r).max()) + 1e-3
        rec["max_err_" + name] = err
        rec["max_ref_" + name] = float(np.abs(r).max())
        ok = ok and err <= lim
    rec["pass"] = ok
    return rec


def bwd_record(args, w, device, dist, world, rank):
    """Measure the backward pass on workload w (see the module docstring)."""
    import oracle
    import warp_specialized_attention_gb300 as wsa
    if w.dtype == "e4m3":
        raise SystemExit("the backward pass takes 16-bit inputs")
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
    enqueue_us = _enqueue_us(step, stream, device)
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

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qh, kh, vh, doh = (t[0, 0].double().cpu().numpy() for t in (q, k, v, d_o))
        t0 = time.perf_counter()
        ref = oracle.attention_bwd(qh, kh, vh, doh, w.causal, w.scale)
        dt = time.perf_counter() - t0
        cpu = {"value": 2.5 * w.flops / (w.B * w.H) / dt / 1e12, "unit": UNIT,
               "cores": oracle.threads(), "kind": "oracle",
               "sample": "one whole (batch, head) slice of %s, backward oracle, %.2f s"
                         % (w.describe(), dt)}
        got = [t[0, 0].double().cpu().numpy() for t in (dq, dk, dv)]
        parity = bwd_parity(w, got, ref)
        parity["sample"] = ("slice (0, 0) of the last timed launch's dQ, dK, dV against the "
                            "backward oracle on the same inputs")

    # e2e: inputs in from pinned host memory, gradients out, every step, through
    # fmha_bwd_host (chunks of (batch, head) slices, copies overlapping the work)
    hin = [t.cpu().pin_memory() for t in (q, k, v, o, lse, d_o)]
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    h2d_gbs, d2h_gbs = _host_link(list(zip(hin, (q, k, v, o, lse, d_o))),
                                  list(zip(hout, (dq, dk, dv))), stream, device)
    del ws
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
    if rank != 0:
        return None
    return {
        "metric": metric_for(w, "bwd"), "value": value,
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(_config(w, in_bytes, flushed), **{"pass": "backward"}),
        "e2e": {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world,
                "ms_per_step": e2e_ms, "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                "link_ms": max(h2d / h2d_gbs, d2h / d2h_gbs) / 1e6,
                "api": "fmha_bwd_host, pinned host buffers, %s chunks" % (args.chunks or 16)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": _traffic(w.name + "_bwd", KERNEL_SOURCES + BWD_SOURCES),
                     "peak_source": "%s bf16 burst dense (fp16 nominal ratio 1)" % peak_src,
                     "step_ms_mean": step_ms, "step_ms_min": min(launches),
                     "host_enqueue_us": enqueue_us,
                     "note": "a step is 4 launches (memset, delta, backward, dQ conversion)"},
        "cpu_baseline": cpu,
        "parity": parity,
        "clocks": clocks,
        "clocks_ok": _clocks_ok(clocks),
        "gpu_launches": 3 * args.steps,
    }


# The other records of the default run (N=1): the four smaller forward
# configurations, the 8-bit forward and the backward of the headline shape.
EXTRA_CONFIGS = [(w.name, "fwd") for w in synthetic.WORKLOADS[:4]] + \
                [(w.name, "fwd") for w in synthetic.FP8_WORKLOADS] + \
                [(synthetic.HEADLINE.name, "bwd")]

CPU_SECONDS_HEADLINE = 12.0
CPU_SECONDS_EXTRA = 3.0


def _summary(rec):
    """The fields of a record kept under the headline line's `configs`."""
    keep = ("metric", "value", "unit", "ms_per_step", "dtype", "config", "e2e", "roofline",
            "cpu_baseline", "parity", "clocks", "clocks_ok", "gpu_launches", "steps")
    return {k: rec[k] for k in keep if k in rec}


def run_ours(args, w):
    import warp_specialized_attention_gb300 as wsa
    world, rank, local = _dist_env()
    dist = _init_dist(world)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the attention path has no CPU fallback)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wsa.load_library()
    if args.pass_ == "bwd":
        line = bwd_record(args, w, device, dist, world, rank)
    else:
        line = fwd_record(args, w, device, dist, world, rank, CPU_SECONDS_HEADLINE)
    torch.cuda.empty_cache()
    extras = (args.configs == "all" and world == 1 and args.pass_ == "fwd"
              and w.name == synthetic.HEADLINE.name and args.batch is None)
    if extras and line is not None:
        configs = {}
        for name, pass_ in EXTRA_CONFIGS:
            wx = synthetic.by_name(name)
            key = name if pass_ == "fwd" else name + "_bwd"
            if pass_ == "bwd":
                rec = bwd_record(args, wx, device, dist, world, rank)
            else:
                rec = fwd_record(args, wx, device, dist, world, rank, CPU_SECONDS_EXTRA)
            torch.cuda.empty_cache()
            configs[key] = _summary(rec)
        line["configs"] = configs
        line["gpu_launches"] = args.steps
    if dist is not None:
        dist.destroy_process_group()
    if line is not None:
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
    ap.add_argument("--configs", choices=["all", "none"], default="all",
                    help="with the default headline workload at N=1: also measure every "
                         "other named configuration (all, default) or only the headline")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 untimed warm-up steps
    w = synthetic.by_name(args.workload)
    if args.batch is not None:
        w = dataclasses.replace(w, B=args.batch, name="%s_b%d" % (w.name, args.batch))
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
