"""Multi-rank host logic of bench.py on the CPU: two gloo ranks (replicas).

The path shards without exchange, so the only cross-rank steps are the
barrier, the MAX reduction of the step time and the whole-job aggregate; the
reference arm runs on rank 0 alone.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.5, 4.0][rank]
        dist.barrier()
        job_ms = bench.max_over_ranks(ms, world)
        value = bench.whole_job_tflops(1.0e12, world, job_ms)

        class Args:
            steps, warmup, cpu_seconds = 1, 0, 0.1
        ref = bench.run_reference(Args, rank, world) if rank != 0 else "rank0-skipped"
        out.put((rank, job_ms, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job_ms, value, ref in res:
        assert job_ms == 4.0                       # MAX over ranks
        assert value == pytest.approx(2.0 * 1.0e12 / 4e-3 / 1e12)  # 2 replicas' work in the slowest time
    assert res[1][3] is None                       # reference arm: only rank 0 works


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_tflops(2.0e12, 1, 1.0) == pytest.approx(2000.0)
