"""The N > 1 path of bench.py, on the CPU with two gloo ranks: per-rank
workloads (weak scaling: independent (batch, head) slices, no data-path
collective), the max-over-ranks timing and the whole-job value, and the
reference arm's rank-0-only rule."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synthetic


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synthetic.HEADLINE
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        slowest = bench._max_over_ranks(dist, local_ms, None)
        seed = bench.rank_seed(w, rank)
        # each rank's inputs are its own draw (small shape, same recipe)
        qk = synthetic.make_inputs(w, B=1, H=1, S=8, D=8, seed=seed)[0]
        gathered = [torch.zeros_like(qk.float()) for _ in range(world)]
        dist.all_gather(gathered, qk.float())
        q.put((rank, slowest, seed, bool(torch.equal(gathered[0], gathered[1])),
               bench.job_tflops(w, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling_and_max_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, slow0, seed0, same0, v0), (r1, slow1, seed1, same1, v1) = res
    assert slow0 == slow1 == 15.0                      # both report the slowest rank
    assert seed0 != seed1 and not same0 and not same1  # ranks draw different batches
    w = synthetic.HEADLINE
    assert v0 == v1 == pytest.approx(2 * w.flops / 15e-3 / 1e12)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = bench.main.__globals__["argparse"].Namespace(steps=1, warmup=3, gpus=2)
    assert bench.run_reference(args, synthetic.HEADLINE) == 0
    assert capsys.readouterr().out == ""
