"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each running
its own replica; the step time is the max over ranks and the throughput counts
both replicas. No data-path collective exists (requests are independent)."""
import os
import socket

import numpy as np
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


def test_reference_plan_keeps_whole_steps_within_budget():
    # 4.6 s steps: the requested 5 + 20 fit in 150 s and are kept
    assert bench.reference_plan(4.6, 20, 5, 150.0) == (5, 20)
    # slow steps: fewer, but at least one warm-up and one timed whole step
    assert bench.reference_plan(30.0, 20, 5, 150.0) == (1, 4)
    assert bench.reference_plan(500.0, 20, 5, 150.0) == (1, 1)
    w, k = bench.reference_plan(0.01, 1000, 20, 150.0)
    assert (w, k) == (20, 1000)


def test_reference_arm_times_whole_steps(capsys):
    import json

    class A:
        gpus, steps, warmup, workload, ref_budget = 1, 2, 3, "b1_ctx4k", 60.0
    bench.run_reference(A(), rank=0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] >= 1 and line["warmup"] >= 1
    assert abs(line["ms_per_step"] * line["steps"] / 1e3 - line["timed_seconds"]) < 1e-6
    assert "whole steps" in line["cpu_baseline"]["sample"]


def test_byte_model_follows_formats_and_measured_union():
    import gen

    class W:
        def __init__(self, key_fmt, lat_fmt, ctx, n_q):
            self.key_fmt, self.lat_fmt, self.ctx, self.n_q, self.batch = key_fmt, lat_fmt, ctx, n_q, len(ctx)
    # one query per request: 132 B per key, 576 B per selected latent, 217,216 B of q/w/out
    w = W("fp8", "fp8", [1 << 20, 3000], 1)
    assert bench.step_bytes(w, [2048, 2048]) == 132 * ((1 << 20) + 3000) + 576 * 4096 + 2 * 217216
    assert bench.indexer_bytes(w) == 132 * ((1 << 20) + 3000) + 2 * (32 * 128 * 2 + 32 * 4)
    # FP4 formats: 68 B keys read once per request, 352 B latents of the union of its rows' sets
    w4 = W("mxfp4", "nvfp4", [1 << 18], 6)
    assert gen.KEY_BYTES["mxfp4"] == 68 and gen.LAT_BYTES["nvfp4"] == 352
    assert bench.step_bytes(w4, [5000]) == 68 * (1 << 18) + 352 * 5000 + 6 * 217216
    assert bench.step_dtype(w4) != bench.step_dtype(w)
    # the union is counted from the indices a step produced (-1 padding ignored)
    idx = np.array([[0, 5, 9, -1], [5, 9, 11, 12],     # request 0: rows 0, 1
                    [1, 2, -1, -1], [2, 3, -1, -1]],   # request 1
                   np.int32)
    assert bench.latent_union(idx, 2, 2) == [5, 3]
