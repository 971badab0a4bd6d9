"""The benchmark's multi-rank host logic on CPU: world_size 2 over gloo on 127.0.0.1.

With N GPUs, bench.py runs one rank per GPU, each on its own copy of the workload (the
method's (b, h, query-tile) units are independent; no data-path collective), and reports
the whole job's throughput over the slowest rank's time. These tests run the same
reduction with the gloo backend in two spawned CPU processes, and check that the
reference arm does its work on rank 0 only.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 1 + r ms in the kernel leg and 5 - r ms end to end
        ms, e2e = bench.max_over_ranks([1.0 + rank, 5.0 - rank], dist, "cpu")
        dist.barrier()
        queue.put((rank, ms, e2e))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == [(0, 2.0, 5.0), (1, 2.0, 5.0)]


def test_job_throughput_counts_every_rank():
    import bench
    assert bench.job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)
    assert bench.job_tflops(2e12, 4, 2.0) == pytest.approx(4000.0)   # 4 ranks' work in the slowest rank's 2 ms


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    from dense_attention_forward_fwd_gb300.configs import by_name
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(bench.parse(), by_name("tiny-256")) == 0   # returns at once on rank 1
