"""Benchmark of the fused DSA decode step (lightning indexer -> exact top-2048 ->
sparse MLA) through libdsa on synthetic data, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one dsa_decode over the whole batch of the workload (one layer).
Default workload: b4_ctx1m (4 requests x 1,048,576-token context, FP8 index keys
and latents, 64-token pages, random block tables) -- the long-context,
bandwidth-bound case. Its inputs (2.97 GB per step) are larger than the 129 MB
L2, so consecutive steps are timed back to back with no flush.

Multi-GPU (torchrun): every rank runs its own replica of the workload on its
own GPU (requests are independent; no data-path collective); the step time is
the max over ranks and `value` counts the layer-steps of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA decode layer-steps/sec and achieved HBM GB/s (% of GB300 roofline)"
UNIT = "layer-steps/s"
# q_idx bf16 [32][128] + w fp32 [32] + q bf16 [96][576] + out bf16 [96][512] per query row
Q_OUT_B = 32 * 128 * 2 + 32 * 4 + 96 * 576 * 2 + 96 * 512 * 2


def fmt_bytes(inp):
    """Bytes per token of the workload's index key and latent formats."""
    import gen

    return gen.KEY_BYTES[inp.key_fmt], gen.LAT_BYTES[inp.lat_fmt]


def latent_union(idx, batch, n_q):
    """|union over t of S_{b,t}| per request, from the top-k indices a step produced
    (int32 [batch * n_q, K], -1 padded)."""
    idx = np.asarray(idx).reshape(batch, n_q, -1)
    return [int(np.unique(r[r >= 0]).size) for r in idx.reshape(batch, -1)]


def step_bytes(inp, union):
    """Algorithmic bytes of one step: every visible index key once per request, each
    latent of the union of the request's selected sets once, q/w/out per row."""
    kb, lb = fmt_bytes(inp)
    return sum(kb * int(c) + lb * int(u) + inp.n_q * Q_OUT_B for c, u in zip(inp.ctx, union))


def indexer_bytes(inp):
    """Algorithmic bytes of the indexer stage: keys + scales once, the query and weights."""
    kb, _ = fmt_bytes(inp)
    return sum(kb * int(c) for c in inp.ctx) + inp.batch * inp.n_q * (32 * 128 * 2 + 32 * 4)


def step_dtype(inp):
    """The arithmetic of the step: the scorer's MMA operands and the attention MMA's."""
    storage = {"fp8": "fp8", "mxfp4": "mxfp4"}[inp.key_fmt] + "/" + {"fp8": "fp8", "nvfp4": "nvfp4"}[inp.lat_fmt]
    return "fp8+bf16" if storage == "fp8/fp8" else f"fp8+bf16 ({storage} storage)"


PROFILE_DIR = os.path.join(ROOT, "profiles")
INDEXER_SOURCES = ("indexer.cu", "sm103_ptx.cuh", "dsa_internal.cuh")


def indexer_source_hash() -> str:
    import hashlib

    h = hashlib.sha256()
    for f in INDEXER_SOURCES:
        with open(os.path.join(ROOT, "dsa_sparse_mla_paged_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def indexer_traffic(workload: str):
    """DRAM bytes per launch of the indexer stage (its two kernels) from the committed
    ncu summary of this workload, or None when the summary was taken on other
    indexer sources than the ones built now."""
    path = os.path.join(PROFILE_DIR, f"indexer_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("indexer_source_sha256_16") != indexer_source_hash():
        return None
    try:
        return int(vals["stage_dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest of each rank's value (the slowest rank sets the step time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(ms_per_step: float, world: int) -> float:
    """Layer-steps/s of the whole job: every rank runs one replica step per ms_per_step."""
    return world * 1e3 / ms_per_step


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(inp, budget_s=15.0):
    """The oracle, as it stands, on whole requests of the workload until ~budget_s."""
    from oracle import dsa as O

    t0 = time.perf_counter()
    done = 0
    for b in range(inp.batch):
        O.decode(inp, requests=[b])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    per_step = dt / done * inp.batch
    return {"value": 1.0 / per_step, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{done} of {inp.batch} requests of one step (numpy float64; BLAS threads = default)",
            "seconds": dt, "single_thread_b1_ctx4k_s": oracle_single_thread_small()}


def oracle_single_thread_small():
    """Seconds of the oracle's whole step on the small parity workload (b1_ctx4k),
    in a fresh interpreter limited to one BLAS / OpenMP thread."""
    code = ("import sys, time; sys.path.insert(0, %r); import gen; from oracle import dsa as O; "
            "inp = gen.make_workload('b1_ctx4k'); t = time.perf_counter(); O.decode(inp); "
            "print(time.perf_counter() - t)") % ROOT
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=300)
        return float(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None


def reference_plan(t_step, steps, warmup, budget_s):
    """Whole oracle steps to run: (warm-up steps, timed steps) within budget_s seconds,
    given the seconds of one step. The requested counts are kept when they fit; at
    least one of each is run."""
    w = max(1, min(warmup, int(0.2 * budget_s / t_step)))
    k = max(1, min(steps, int(0.8 * budget_s / t_step)))
    return w, k


def run_reference(args, rank):
    """The reference arm: the oracle (float64 NumPy on the host cores) running whole
    steps of the workload -- every request of the batch per step."""
    import gen

    line = {"impl": "reference", "metric": METRIC, "unit": UNIT, "higher_is_better": True, "n_gpus": args.gpus,
            "data": "synthetic", "scaling": "weak", "vs_baseline": None, "dtype": "f64"}
    if rank != 0:
        return
    from oracle import dsa as O

    inp = gen.make_workload(args.workload)
    t0 = time.perf_counter()
    O.decode(inp)  # the first warm-up step, which also sizes the run
    t_first = time.perf_counter() - t0
    warm, steps = reference_plan(t_first, args.steps, args.warmup, getattr(args, "ref_budget", 150.0))
    for _ in range(warm - 1):
        O.decode(inp)
    t0 = time.perf_counter()
    for _ in range(steps):
        O.decode(inp)
    dt = time.perf_counter() - t0
    per_step = dt / steps
    v = 1.0 / per_step
    cores = len(os.sched_getaffinity(0))
    line.update({"steps": steps, "warmup": warm, "steps_requested": args.steps, "warmup_requested": args.warmup,
                 "value": v, "ms_per_step": per_step * 1e3, "timed_seconds": dt,
                 "config": {"workload": args.workload, "batch": inp.batch, "n_q": inp.n_q,
                            "ctx": int(inp.ctx.max()), "topk": inp.topk},
                 "cpu_baseline": {"value": v, "unit": UNIT, "kind": "oracle", "cores": cores,
                                  "sample": f"{steps} whole steps ({inp.batch} requests each), timed back to back"},
                 "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})
    print(json.dumps(line), flush=True)


def run_stage(args):
    """Time one entry point alone (for kernel profiles):
    `--stage indexer|topk|mla|dcp_merge|dcp_combine|frontend|prefill` (the front end with
    d_c = 1536, d_model = 7168 and its weights rotated through 12 copies, 173 MB > L2;
    prefill: rank --rank of --world token slices, e.g. on --workload b1_prefill2k_ctx150k)."""
    import torch

    import dsa_sparse_mla_paged_gb300 as dsa
    import gen

    from gen.device import Dev

    torch.cuda.set_device(0)
    dsa.load()
    inp = gen.make_workload(args.workload)
    d = Dev(inp)
    sc = torch.empty((d.rows, d.cap), dtype=torch.float32, device="cuda")
    idx = torch.empty((d.rows, inp.topk), dtype=torch.int32, device="cuda")
    out = torch.empty((d.rows, 96, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((d.rows, 96), dtype=torch.float32, device="cuda")
    # inputs of the later stages come from the earlier ones, computed once untimed
    dsa.indexer_scores(d.p, d.q_idx, d.w, d.key_pool, d.block_table, d.ctx, sc, d.cap, d.ws)
    dsa.topk(d.p, sc, d.cap, d.ctx, d.block_table, idx, None, d.ws)
    W = args.world
    stats = torch.zeros((d.rows, 2), dtype=torch.int32, device="cuda")
    # the front end's weights, in enough copies that the rotation exceeds L2
    D_C, D_MODEL = 1536, 7168
    fe_copies = 12 if args.stage == "frontend" else 1
    gen_ = torch.Generator(device="cuda").manual_seed(9)
    fe_wq = [torch.randn((4096, D_C), device="cuda", generator=gen_).mul_(D_C ** -0.5).bfloat16()
             for _ in range(fe_copies)]
    fe_wk = [torch.randn((128, D_MODEL), device="cuda", generator=gen_).mul_(D_MODEL ** -0.5).bfloat16()
             for _ in range(fe_copies)]
    fe_cq = torch.randn((d.rows, D_C), device="cuda", generator=gen_).bfloat16()
    fe_g = torch.ones(D_C, device="cuda").bfloat16()
    fe_x = torch.randn((d.rows, D_MODEL), device="cuda", generator=gen_).bfloat16()
    fe_w = torch.rand((d.rows, 32), device="cuda", generator=gen_)
    fe_dims = dsa.FrontendDims(d_c=D_C, d_model=D_MODEL, eps=1e-6)
    fe_i = [0]

    def fe_call():
        k = fe_i[0] % fe_copies
        fe_i[0] += 1
        dsa.indexer_frontend(d.p, fe_dims, fe_cq, fe_g, fe_wq[k], fe_w, fe_x, fe_wk[k], d.key_pool, d.block_table,
                             d.ctx, d.ws)
    parts_o = torch.zeros((W, d.rows, 96, 512), dtype=torch.bfloat16, device="cuda")
    parts_l = torch.zeros((W, d.rows, 96), dtype=torch.float32, device="cuda")
    calls = {
        "indexer": lambda: dsa.indexer_scores(d.p, d.q_idx, d.w, d.key_pool, d.block_table, d.ctx, sc, d.cap, d.ws),
        "dcp_merge": lambda: dsa.dcp_topk_merge(d.p, sc, d.cap, d.ctx, W, idx, stats, d.ws),
        "dcp_combine": lambda: dsa.lse_combine(d.p, W, parts_o, parts_l, out, lse),
        "frontend": lambda: fe_call(),
        "prefill": lambda: dsa.indexer_prefill_scores(d.p, W, max(args.rank, 0), d.q_idx, d.w, d.key_pool,
                                                      d.block_table, d.ctx, sc, d.cap, d.ws),
        "topk": lambda: dsa.topk(d.p, sc, d.cap, d.ctx, d.block_table, idx, None, d.ws),
        "mla": lambda: dsa.sparse_mla_decode(d.p, d.q, d.lat_pool, d.block_table, d.ctx, idx, out, lse, d.ws),
    }
    f = calls[args.stage]
    if args.stage == "prefill" and args.rank < 0:
        # every rank of the token split in turn: the balance of the r / 2W-1-r pairing
        per_rank = []
        for r in range(W):
            args.rank = r
            for _ in range(args.warmup):
                f()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(args.steps):
                f()
            e1.record()
            torch.cuda.synchronize()
            per_rank.append(e0.elapsed_time(e1) / args.steps)
        args.rank = -1
        print(json.dumps({"stage": "prefill", "workload": args.workload, "world": W,
                          "ms_per_rank": per_rank, "max_over_min": max(per_rank) / min(per_rank)}), flush=True)
        return
    for _ in range(args.warmup):
        f()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record()
    for _ in range(args.steps):
        f()
    ev1.record()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / args.steps
    score_bytes = 4 * sum(int(c) for c in inp.ctx) * inp.n_q
    nbytes = {"indexer": indexer_bytes(inp), "topk": score_bytes,
              "mla": step_bytes(inp, latent_union(idx.cpu().numpy(), inp.batch, inp.n_q)) - indexer_bytes(inp),
              # every score read once; the partials read once and the result written
              "dcp_merge": score_bytes, "dcp_combine": (W + 1) * d.rows * 96 * 512 * 2 + (W + 1) * d.rows * 96 * 4,
              # weights once, the rows' inputs, q8 + w' out, one key per row
              "frontend": (4096 * D_C + 128 * D_MODEL + D_C) * 2 + d.rows * ((D_C + D_MODEL) * 2 + 32 * 4)
                          + d.rows * (4096 + 32 * 4 + 132),
              "prefill": 0,
              }[args.stage]
    assert dsa.get_device_error(d.ws) == 0
    line = {"stage": args.stage, "workload": args.workload, "ms": ms, "bytes": nbytes,
            "gbs": nbytes / (ms * 1e-3) / 1e9}
    if args.stage == "prefill":
        # useful work of the scored rows: every visible key of every row, 32 heads x 128 dims
        rows = list(range(inp.n_q)) if W == 1 else [int(t) for t in _rank_rows(inp.n_q, W, max(args.rank, 0))]
        keys = sum(max(0, int(c) - inp.n_q + t + 1) for c in inp.ctx for t in rows)
        flops = 2.0 * 32 * 128 * keys
        byts = fmt_bytes(inp)[0] * sum(int(c) for c in inp.ctx) + 4 * keys + len(rows) * inp.batch * (32 * 128 * 2 + 32 * 4)
        line.update({"world": W, "rank": max(args.rank, 0), "rows_scored": len(rows) * inp.batch,
                     "keys_scored": keys, "bytes": byts, "gbs": byts / (ms * 1e-3) / 1e9,
                     "tflops": flops / (ms * 1e-3) / 1e12})
    if args.stage == "dcp_merge":
        st = stats.cpu().numpy()
        full = W * inp.topk * 8  # every shard's local top-K as (fp32 score, int32 token) pairs
        line.update({"world": W, "resent_rows": int((st[:, 0] != 0).sum()),
                     "words_per_row": [int(x) for x in st[:, 1]],
                     "traffic_ratio_vs_full_exchange": [full / (4 * int(x)) for x in st[:, 1]]})
        line["cpu_baseline"] = cpu_baseline_dcp(sc[0, :int(inp.ctx[0]) - inp.n_q + 1].cpu().numpy(), W, inp.topk,
                                                idx[0].cpu().numpy())
    print(json.dumps(line), flush=True)


def cpu_baseline_dcp(row, world, topk, gpu_idx):
    """The oracle's merge of one row of the same scores, timed on the host (the
    stage's CPU baseline), and whether the GPU's row equals it."""
    from oracle import dcp as D

    t0 = time.perf_counter()
    res = D.merge(row, world, topk)
    dt = time.perf_counter() - t0
    return {"kind": "oracle", "sample": "row 0 of the call", "ms_per_row": dt * 1e3,
            "cores": len(os.sched_getaffinity(0)), "row0_equals_gpu": bool(np.array_equal(gpu_idx, res["idx"]))}


def _rank_rows(n_q, world, rank):
    """Rows of one request that rank `rank` of `world` scores (slices r and 2W - 1 - r of 2W)."""
    ss = n_q // (2 * world)
    return list(range(rank * ss, (rank + 1) * ss)) + list(range((2 * world - 1 - rank) * ss, (2 * world - rank) * ss))


def run_ours(args, rank, world):
    import torch

    import dsa_sparse_mla_paged_gb300 as dsa
    import gen

    from gen.device import Dev

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dsa.load()

    inp = gen.make_workload(args.workload)
    cpu = cpu_baseline(inp) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    d = Dev(inp)
    stream = torch.cuda.Stream()
    out = torch.empty((d.rows, 96, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((d.rows, 96), dtype=torch.float32, device="cuda")
    idx = torch.empty((d.rows, inp.topk), dtype=torch.int32, device="cuda")

    def step(s):
        dsa.decode(d.p, d.q_idx, d.w, d.key_pool, d.q, d.lat_pool, d.block_table, d.ctx, out, lse, idx, d.ws,
                   stream=s)

    # Parts of the same step for the live kernel timing: [indexer stage] and
    # [top-k + attention], each through its stage entry point and captured in a
    # CUDA graph of its own.
    sc = torch.empty((d.rows, d.cap), dtype=torch.float32, device="cuda")

    def part_indexer(s_):
        dsa.indexer_scores(d.p, d.q_idx, d.w, d.key_pool, d.block_table, d.ctx, sc, d.cap, d.ws, stream=s_)

    def part_rest(s_):
        dsa.topk(d.p, sc, d.cap, d.ctx, d.block_table, idx, None, d.ws, stream=s_)
        dsa.sparse_mla_decode(d.p, d.q, d.lat_pool, d.block_table, d.ctx, idx, out, lse, d.ws, stream=s_)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            step(stream)
            part_indexer(stream)
            part_rest(stream)
    stream.synchronize()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn(torch.cuda.current_stream())
        return g

    graph = capture(step)
    parts = [capture(part_indexer), capture(part_rest)]
    torch.cuda.synchronize()
    if dsa.get_device_error(d.ws) != 0:
        raise RuntimeError("device error word set during warm-up")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
            parts[0].replay()
            parts[1].replay()
    barrier()
    # The timed region: K steps of dsa_decode replayed from one graph, then the
    # same K steps replayed as the two parts with an event pair around the
    # indexer stage of every step (events on the launching stream), which times
    # the dominant kernel live. The step time reported is the first loop's.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.15)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
            for i in range(args.steps):
                ev_a[i].record(stream)
                parts[0].replay()
                ev_b[i].record(stream)
                parts[1].replay()
            ev_end.record(stream)
        barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, "cuda")
    ms_parts = max_over_ranks(ev_a[0].elapsed_time(ev_end) / args.steps, dist, "cuda")
    idx_ms_live = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / args.steps, dist, "cuda")

    # per-stage times: each stage entry point captured in its own CUDA graph and
    # replayed back to back (events on the launching stream; no host overhead)
    stage_calls = {
        "indexer": part_indexer,
        "topk": lambda s_: dsa.topk(d.p, sc, d.cap, d.ctx, d.block_table, idx, None, d.ws, stream=s_),
        "sparse_mla": lambda s_: dsa.sparse_mla_decode(d.p, d.q, d.lat_pool, d.block_table, d.ctx, idx, out, lse,
                                                       d.ws, stream=s_),
    }
    stage_ms = {}
    nst = max(10, min(args.steps, 200))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with torch.cuda.stream(stream):
        for name, call in stage_calls.items():
            call(stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(torch.cuda.current_stream())
            for _ in range(3):
                g.replay()
            ev[0].record(stream)
            for _ in range(nst):
                g.replay()
            ev[1].record(stream)
            stream.synchronize()
            stage_ms[name] = ev[0].elapsed_time(ev[1]) / nst

    # End to end through the public call, host buffers, copies inside the timed
    # region: the step's inputs (q_idx, w, q, block table, context lengths) sit
    # in one pinned host buffer and travel in one copy to one device buffer whose
    # pieces dsa_decode reads; its results (out, lse) come back in one copy to a
    # pinned host buffer. As a serving loop would, two buffer sets alternate so
    # that step i + 1's inputs and step i - 1's results cross while step i
    # computes: copies on a second stream, dsa_decode (a CUDA graph per buffer
    # set) on the first, ordered by events.
    ins = [d.q_idx, d.w, d.q, d.block_table, d.ctx]
    offs, o = [], 0
    for t in ins:
        offs.append(o)
        o = (o + t.numel() * t.element_size() + 255) // 256 * 256
    piece = lambda buf, off, t: buf[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
    o_off = (out.numel() * out.element_size() + 255) // 256 * 256
    h_in = torch.empty(o, dtype=torch.uint8).pin_memory()
    for t, off in zip(ins, offs):
        piece(h_in, off, t).copy_(t.cpu())
    bufs = []
    for _ in range(2):
        d_in = torch.empty(o, dtype=torch.uint8, device="cuda")
        d_out = torch.empty(o_off + lse.numel() * 4, dtype=torch.uint8, device="cuda")
        h_out = torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory()
        views = [piece(d_in, off, t) for t, off in zip(ins, offs)]
        bufs.append({"d_in": d_in, "d_out": d_out, "h_out": h_out, "views": views,
                     "out": piece(d_out, 0, out), "lse": piece(d_out, o_off, lse)})
    h2d, d2h = int(h_in.numel()), int(bufs[0]["h_out"].numel())
    in_st, out_st = torch.cuda.Stream(), torch.cuda.Stream()

    def decode_into(bf, s_):
        e_q_idx, e_w, e_q, e_bt, e_ctx = bf["views"]
        dsa.decode(d.p, e_q_idx, e_w, d.key_pool, e_q, d.lat_pool, e_bt, e_ctx, bf["out"], bf["lse"], idx, d.ws,
                   stream=s_)

    for bf in bufs:
        with torch.cuda.stream(stream):
            bf["d_in"].copy_(h_in)
            decode_into(bf, stream)
            stream.synchronize()
            bf["graph"] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(bf["graph"], stream=stream):
                decode_into(bf, torch.cuda.current_stream())
        bf["ev_in"], bf["ev_done"], bf["ev_out"] = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()

    def run_e2e(n):
        # inputs in on in_st, the step on `stream`, results out on out_st
        for i in range(n):
            bf = bufs[i & 1]
            in_st.wait_event(bf["ev_done"])  # step i - 2 has read these inputs
            with torch.cuda.stream(in_st):
                bf["d_in"].copy_(h_in, non_blocking=True)
            bf["ev_in"].record(in_st)
            stream.wait_event(bf["ev_in"])
            stream.wait_event(bf["ev_out"])  # step i - 2's results have left
            with torch.cuda.stream(stream):
                bf["graph"].replay()
            bf["ev_done"].record(stream)
            out_st.wait_event(bf["ev_done"])
            with torch.cuda.stream(out_st):
                bf["h_out"].copy_(bf["d_out"], non_blocking=True)
            bf["ev_out"].record(out_st)
        stream.wait_stream(out_st)

    torch.cuda.synchronize()
    for bf in bufs:
        bf["ev_done"].record(stream)
        bf["ev_out"].record(stream)
    run_e2e(4)
    torch.cuda.synchronize()
    for bf in bufs:
        assert torch.equal(piece(bf["h_out"], 0, out), out.cpu()), "the end-to-end step must give the fused step's output"
    ke2e = max(6, min(args.steps, 100))
    barrier()
    ev[0].record(stream)
    in_st.wait_event(ev[0])
    run_e2e(ke2e)
    ev[1].record(stream)
    barrier()
    e2e_ms = max_over_ranks(ev[0].elapsed_time(ev[1]) / ke2e, dist, "cuda")

    if rank == 0:
        peak, peak_kind = peaks()
        union = latent_union(idx.cpu().numpy(), inp.batch, inp.n_q)
        sbytes = step_bytes(inp, union)
        ibytes = indexer_bytes(inp)
        gbs = sbytes / (ms * 1e-3) / 1e9
        idx_gbs = ibytes / (idx_ms_live * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": replica_throughput(ms, world), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": step_dtype(inp), "data": "synthetic",
            "config": {"workload": args.workload, "batch": inp.batch, "n_q": inp.n_q,
                       "ctx": int(inp.ctx.max()), "topk": inp.topk, "page_size": inp.page_size,
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (%.2f GB per step), no flush" % (
                           (inp.key_pool.nbytes + inp.lat_pool.nbytes) / 1e9)},
            "achieved_gbs": gbs, "hbm_frac": gbs / peak, "step_bytes": sbytes,
            "latent_union_per_request": {"min": min(union), "max": max(union), "sum": sum(union)},
            "stage_ms": stage_ms, "ms_per_step_as_parts": ms_parts,
            "roofline": {"bound": "hbm", "kernel": "indexer stage (dsa_indexer_scores: q quantisation + scorer)",
                         "achieved": idx_gbs,
                         "peak": peak, "unit": "GB/s", "frac": idx_gbs / peak,
                         "traffic": indexer_traffic(args.workload),
                         "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": ibytes,
                         "launch_ms": idx_ms_live},
            "e2e": {"value": replica_throughput(e2e_ms, world), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * args.steps * dsa.KERNELS_PER_DECODE,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="b4_ctx1m")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=150.0,
                    help="reference arm: seconds of oracle steps to run at most (warm-up + timed)")
    ap.add_argument("--stage", default="all",
                    choices=["all", "indexer", "topk", "mla", "dcp_merge", "dcp_combine", "frontend", "prefill"],
                    help="time one entry point alone (kernel profiling; the dcp_* stages emulate --world shards)")
    ap.add_argument("--world", type=int, default=8, help="shards of the dcp_* stages, ranks of the prefill stage")
    ap.add_argument("--rank", type=int, default=0, help="prefill stage: this rank's slices (-1: every rank in turn)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
    elif args.stage != "all":
        run_stage(args)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
