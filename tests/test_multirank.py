"""The multi-GPU mode of bench.py (independent replicas, one per rank: the
layer has no exchange step) on the CPU with gloo ranks, world size 2: the
host-side logic only -- replica batches, the max-over-ranks time, the
whole-job throughput, and the reference arm's rank-0-only rule."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from sparse_mixture_experts_51_b300 import workloads as W


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 40.0][rank]
        got = bench.max_over_ranks(local_ms, world)
        w = bench.replica_workload(W.WORKLOADS["tiny_fp32"], rank, world)
        x = W.make_inputs(w)["x"]
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, x.double().sum().reshape(1))
        dist.barrier()
        out[rank] = (got, w.seed, float(sums[0]), float(sums[1]))
    finally:
        dist.destroy_process_group()


def test_replicas_on_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    (m0, s0, a0, b0), (m1, s1, a1, b1) = out[0], out[1]
    assert m0 == m1 == 40.0                      # every rank sees the slowest rank's time
    assert s0 != s1                              # independent token batches
    assert a0 == a1 and b0 == b1 and a0 != b0    # and both ranks agree on what each drew


def test_job_throughput_counts_every_rank():
    # 2 ranks x 100 steps x 4096 tokens in 50 ms (the slowest rank) -> 16.384 M tokens/s
    assert bench.job_throughput(4096, 100, 2, 50.0) == pytest.approx(16.384e6)
    assert bench.max_over_ranks(3.0, 1) == 3.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    called = []
    monkeypatch.setattr(bench, "cpu_oracle_run", lambda *a, **k: called.append(1) or (1.0, "", 1, 1.0))
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])) == 0
    assert called == []


def test_step_quantiles():
    """Median and nearest-rank 95th percentile of per-step times."""
    v = [float(i) for i in range(1, 21)]
    q = bench.step_quantiles(list(reversed(v)))
    assert q == {"p50": 10.5, "p95": 19.0}
    assert bench.step_quantiles([0.25]) == {"p50": 0.25, "p95": 0.25}
    assert bench.step_quantiles([]) is None
