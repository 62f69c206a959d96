"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each running
its own replica; the step time is the max over ranks and the throughput counts
both replicas. No data-path collective exists (requests are independent)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        q.put((rank, ms, bench.replica_throughput(ms, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [2.5, 2.5]
    assert all(abs(g[2] - 2 * 1e3 / 2.5) < 1e-9 for g in got)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.replica_throughput(0.5, 1) == 2000.0


def test_reference_arm_other_ranks_do_no_work(capsys):
    class A:
        gpus, steps, warmup, workload = 2, 1, 3, "b1_ctx4k"
    bench.run_reference(A(), rank=1)
    assert capsys.readouterr().out == ""
