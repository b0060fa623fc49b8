#!/usr/bin/env python3
"""Benchmark of the copy-on-write tree KV cache hot path on GB300.

Workload (default): Llama-3-8B-shaped attention layer (32 Q heads, 8 KV heads,
head_dim 128, bf16, block_size 16); 8 independent requests with a 4096-token
shared prefix, forked 4 ways, each branch 256 divergent tokens, one decode
query per branch.  The prefixes are prefilled once before timing (resident in
HBM).  One step is one pass of the whole path over that batch:

    fork (8 parents x 4 children, batched)  ->  copy-on-write append of the
    256 divergent tokens of all 32 branches  ->  tree decode attention (plan,
    shared-prefix + leaf partials, log-sum-exp merge)  ->  free of the 32 branches

`value` is branch-queries per second of step time (32 queries per step per
GPU; all ranks summed).  The roofline entry covers the dominant kernel, the
attention partial kernel: unique KV bytes (each shared block counted once)
plus Q read and partial/out bytes excluded, over its CUDA-event duration.

`--impl reference` times the fp64 CPU oracle (single thread) on a bounded
sample of the same workload: the tree attention of the 4 branches of one
request per step.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers

# DRAM bytes (read + write) per launch of k_attn_partial_bf16 on this step,
# from one ncu capture of the kernel as it is now (dram__bytes_read.sum
# 168.27 MB + dram__bytes_write.sum 4.62 MB); to be re-taken whenever that
# kernel changes.
BEAM_PARTIAL_TRAFFIC_BYTES = 172_880_000

def quantile(xs, q):
    """The q-quantile of xs (nearest rank)."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q * (len(ys) - 1)))))]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (a timing reduction, not a data-path
    collective)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBps", "copy_gbs"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi (every 50 ms)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5:
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.proc = None

    def summary(self, t0: float, t1: float):
        """Samples received in [t0, t1 + 0.1 s]; if none, the two nearest."""
        time.sleep(0.12)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ts, ln in list(self.lines):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((ts, float(f[1]), float(f[2]), f[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.1]
        window = "timed region"
        if not inside and rows:
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
            window = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------ workload
def beam_workload(seed: int):
    from copy_write_forked_gb300 import workloads as W
    return W.beam(requests=8, prefix=4096, width=4, divergent=256, seed=seed)


def config_of(w):
    m = w.meta
    return {"workload": "beam-like 4-way fork, Llama-3-8B attention layer", "name": w.name,
            "requests": m["requests"], "prefix_tokens": m["prefix"], "fork_width": m["width"],
            "divergent_tokens": m["divergent"], "branch_queries_per_step": len(w.query),
            "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "l2": "flushed before every step (read-only pass over 256 MiB)",
            "step": "fork + CoW append + tree decode attention + free"}


# ---------------------------------------------------------- our arm
def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__ as g
    g.build()
    from copy_write_forked_gb300.dendrite import Pool
    from copy_write_forked_gb300 import workloads as W

    w = beam_workload(seed=rank)
    R, P, Wd, Dv = (w.meta[k] for k in ("requests", "prefix", "width", "divergent"))
    nq, nkv, d = w.n_q_heads, w.n_kv_heads, w.head_dim
    bs = w.block_size
    nblocks = R * (P // bs + 1) + R * Wd * (Dv // bs + 2) + 64
    pool = Pool(nblocks, bs, nkv, d, torch.bfloat16, max_branches=R * (Wd + 1) + 8,
                max_blocks_per_branch=(P + Dv) // bs + 8)
    # prefill (untimed): the 8 prefixes, resident in HBM
    roots = [pool.new_branch() for _ in range(R)]
    prefill_idx = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == P)
    Kp, Vp = w.kv(prefill_idx, dev)
    pool.append_kv(roots, Kp, Vp)
    del Kp, Vp
    div_idx = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == Dv)
    Kd, Vd = w.kv(div_idx, dev)            # divergent tokens of the 32 branches, resident
    Q = w.q(dev)
    out = torch.empty_like(Q)
    stream = torch.cuda.current_stream()
    pool.sync()

    flush_r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        # read-only pass over 256 MiB (2x L2): evicts the cache and leaves it
        # holding clean lines, so no write-back lands inside the next step
        flush_r.max()

    def step():
        kids = pool.fork_batch(roots, [Wd] * R)
        br = [c for ks in kids for c in ks]
        pool.append_kv(br, Kd, Vd)
        pool.tree_attn_decode(Q, br, out=out)
        pool.free(br)
        return br

    clk = ClockSampler(local).__enter__()
    pool.set_profiling(False)
    for _ in range(args.warmup):
        flush_l2()
        step()
    pool.sync()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    # ---- timed region: K steps enqueued back to back, one event pair per step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_clk0 = time.time()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    t_clk1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.summary(t_clk0, t_clk1)
    clk.__exit__(None, None, None)
    pool.sync()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(step_ms)
    ms = max_over_ranks(ms, world, dev)
    n_queries = len(w.query)
    value = world * n_queries / (ms / 1e3)

    # ---- per-kernel device times (profiling events inside the library; one
    # synchronised step at a time so the events of each call can be read)
    pool.set_profiling(True)
    kern = {k: [] for k in ("fork", "append_meta", "append_copy", "attn_partial", "attn_merge", "free",
                            "attn_total")}
    plan_us = []

    def step_profiled():
        # A second L2 flush sits right before the attention call: the device
        # works through it while the host builds the plan and launches, so the
        # events around the attention kernels time the kernels, not the host.
        kids = pool.fork_batch(roots, [Wd] * R)
        br = [c for ks in kids for c in ks]
        pool.append_kv(br, Kd, Vd)
        flush_l2()
        pool.tree_attn_decode(Q, br, out=out)
        pool.free(br)

    for i in range(min(args.steps, 100)):
        flush_l2()
        step_profiled()
        tm = pool.last_timings()
        plan_us.append(pool.last_plan_stats()["plan_us"])
        for k in kern:
            if tm.get(k) is not None:
                kern[k].append(tm[k])
    pool.set_profiling(False)

    # roofline of the attention partial kernel
    unique_kv = w.unique_kv_bytes()
    q_bytes = Q.numel() * Q.element_size()
    attn_ms = statistics.mean(kern["attn_partial"])
    achieved = (unique_kv + q_bytes) / (attn_ms / 1e3) / 1e9
    peak, peak_src = read_peaks()
    plan = pool.last_plan_stats()

    # ----- e2e through the public API with host buffers (pinned), H2D + D2H inside
    # the timed region.  A copy stream brings step i + 1's K, V and Q in while
    # the compute stream runs step i (two device buffer sets); the result of
    # every step is read back to pinned host memory on the compute stream.
    Kh, Vh, Qh = Kd.cpu().pin_memory(), Vd.cpu().pin_memory(), Q.cpu().pin_memory()
    outh = [torch.empty(Q.shape, dtype=Q.dtype).pin_memory() for _ in range(2)]
    bufs = [(torch.empty_like(Kd), torch.empty_like(Vd), torch.empty_like(Q), torch.empty_like(Q))
            for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer set j landed
    ev_used = [torch.cuda.Event() for _ in range(2)]   # step using buffer set j finished
    for e in ev_used:
        e.record(stream)

    def bring_in(j):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_used[j])
            K2, V2, Q2, _ = bufs[j]
            K2.copy_(Kh, non_blocking=True)
            V2.copy_(Vh, non_blocking=True)
            Q2.copy_(Qh, non_blocking=True)
            ev_in[j].record(copy_stream)

    def e2e_step(j):
        K2, V2, Q2, o2 = bufs[j]
        stream.wait_event(ev_in[j])
        kids = pool.fork_batch(roots, [Wd] * R)
        br = [c for ks in kids for c in ks]
        pool.append_kv(br, K2, V2)
        pool.tree_attn_decode(Q2, br, out=o2)
        outh[j].copy_(o2, non_blocking=True)
        pool.free(br)
        ev_used[j].record(stream)

    def e2e_run(n):
        bring_in(0)
        for i in range(n):
            if i + 1 < n:
                bring_in((i + 1) % 2)
            e2e_step(i % 2)

    for _ in range(args.warmup):
        flush_l2()
        e2e_run(2)
    torch.cuda.synchronize()
    flush_l2()
    torch.cuda.synchronize()
    e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    e2e_ev[0].record(stream)
    copy_stream.wait_stream(stream)
    e2e_run(args.steps)
    stream.wait_stream(copy_stream)
    e2e_ev[1].record(stream)
    torch.cuda.synchronize()
    e2e = max_over_ranks(e2e_ev[0].elapsed_time(e2e_ev[1]) / args.steps, world, dev)
    h2d = (Kh.numel() + Vh.numel() + Qh.numel()) * 2
    d2h = outh[0].numel() * 2
    # the inputs are exact copies, so the last step's output matches the device-resident run's
    if (outh[(args.steps - 1) % 2].to(dev).float() - out.float()).abs().max().item() > 1e-2:
        raise RuntimeError("e2e output differs from the device-resident step")

    # ----- fork latency at depth 500 blocks (tail half full), 1 and 4 children
    fork = fork_latency(dev) if rank == 0 else {}
    pool.sync()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    # fork 1 + append 2 (meta, copy) + attention 3 (the step's new tree needs a new
    # plan: its upload, then partial and merge) + free 1
    gpu_launches = 7 * args.steps
    line = {
        "metric": "tree decode attn branch-queries/s & HBM GB/s (unique KV) vs peak; fork us",
        "value": value, "unit": "branch-queries/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (Q/K/V ~ N(0,1), seeded)",
        "config": dict(config_of(w), parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": {"bound": "hbm", "kernel": "k_attn_partial_bf16", "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": BEAM_PARTIAL_TRAFFIC_BYTES,
                     "algorithmic_bytes": unique_kv + q_bytes, "kernel_ms": attn_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": world * n_queries / (e2e / 1e3), "unit": "branch-queries/s", "ms_per_step": e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "kernels_ms": {k: (statistics.mean(v) if v else None) for k, v in kern.items()},
        "attn_branch_queries_per_s": n_queries / (statistics.mean(kern["attn_total"]) / 1e3),
        "plan": {"segments": plan["n_segments"], "units": plan["n_units"], "ctas": plan["n_ctas"],
                 "partials": plan["n_partials"], "tiles": plan["tiles"], "unique_tiles": plan["unique_tiles"],
                 "host_plan_us_mean": statistics.mean(plan_us)},
        "fork_us": fork,
        "wall_s": wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    pool.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_decode_layers(args):
    """The beam step through all 32 layers of a Llama-3-8B-shaped model: one
    fork, one append_begin (block decisions for every layer), then per layer
    append_layer (that layer's rows) and tree attention over that layer (the
    plan is built for layer 0 and reused), then one free.  Synthetic K/V per
    layer, resident in HBM; L2 flushed before every step."""
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__ as g
    g.build()
    from copy_write_forked_gb300.dendrite import Pool
    NL = 32
    w = beam_workload(seed=rank)
    R, P, Wd, Dv = (w.meta[k] for k in ("requests", "prefix", "width", "divergent"))
    nq, nkv, d, bs = w.n_q_heads, w.n_kv_heads, w.head_dim, w.block_size
    nblocks = R * (P // bs + 1) + R * Wd * (Dv // bs + 2) + 64
    pool = Pool(nblocks, bs, nkv, d, torch.bfloat16, max_branches=R * (Wd + 1) + 8,
                max_blocks_per_branch=(P + Dv) // bs + 8, n_layers=NL)
    roots = [pool.new_branch() for _ in range(R)]
    prefill_idx = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == P)
    div_idx = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == Dv)
    pool.append_begin(roots, P)
    for l in range(NL):
        Kp, Vp = w.kv(prefill_idx, dev, layer=l)
        pool.append_layer(l, Kp, Vp)
        del Kp, Vp
    Kd = [w.kv(div_idx, dev, layer=l) for l in range(NL)]
    Q = w.q(dev)
    outs = [torch.empty_like(Q) for _ in range(NL)]
    stream = torch.cuda.current_stream()
    flush_r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        kids = pool.fork_batch(roots, [Wd] * R)
        br = [c for ks in kids for c in ks]
        pool.append_begin(br, Dv)
        for l in range(NL):
            pool.append_layer(l, Kd[l][0], Kd[l][1])
            pool.tree_attn_decode(Q, br, out=outs[l], layer=l)
        pool.free(br)

    for _ in range(args.warmup):
        flush_r.max()
        step()
    pool.sync()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_r.max()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    step_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    # per-layer attention kernels, one synchronised step
    pool.set_profiling(True)
    kids = pool.fork_batch(roots, [Wd] * R)
    br = [c for ks in kids for c in ks]
    pool.append_begin(br, Dv)
    part, plan_us = [], []
    for l in range(NL):
        pool.append_layer(l, Kd[l][0], Kd[l][1])
        flush_r.max()
        pool.tree_attn_decode(Q, br, out=outs[l], layer=l)
        part.append(pool.last_timings()["attn_partial"])
        plan_us.append(pool.last_plan_stats()["plan_us"])
    pool.free(br)
    pool.set_profiling(False)
    pool.sync()
    unique = w.unique_kv_bytes() + Q.numel() * Q.element_size()
    peak, src = read_peaks()
    pk = statistics.median(part)
    n_queries = len(w.query)
    line = {"metric": "tree decode attn branch-queries/s & HBM GB/s (unique KV) vs peak; fork us",
            "workload": "decode32", "value": n_queries * NL / (step_ms / 1e3), "unit": "branch-layer-queries/s",
            "ms_per_step": step_ms, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16",
            "data": "synthetic (Q/K/V ~ N(0,1), seeded per layer)",
            "config": {"workload": "beam step (8 x 4096 prefix, fork 4, 256 divergent) through 32 layers: "
                                   "fork, append_begin, 32 x (append_layer, tree attention), free",
                       "l2": "flushed before every step"},
            "per_layer_partial_kernel_ms": pk,
            "roofline": {"bound": "hbm", "kernel": "k_attn_partial_bf16", "achieved": unique / (pk / 1e3) / 1e9,
                         "peak": peak, "peak_source": src, "unit": "GB/s",
                         "frac": unique / (pk / 1e3) / 1e9 / peak, "algorithmic_bytes": unique},
            "plan_us_layer0": plan_us[0], "plan_us_other_layers_max": max(plan_us[1:]),
            "gpu_launches_per_step": 1 + 1 + 1 + NL * 3 + 1}   # fork, append metadata, plan upload (layer 0), per layer copy + partial + merge, free
    if rank == 0:
        print(json.dumps(line), flush=True)
    pool.close()



def other_workload(name):
    from copy_write_forked_gb300 import workloads as W
    if name == "mcts":
        return W.mcts(), "MCTS tree: root 2048, 500 iterations of fork 4 x 32 tokens, one query per live leaf"
    if name == "specverify":
        return W.spec_verify(), "speculative verification: 32 x prefix 8192, 3 draft paths x 8 tokens, q_len 8"
    if name == "stress":
        return W.fork_stress_attention(), "stress: 16 x prefix 32768, fork 64 x 1024 tokens"
    raise ValueError(name)


def run_attention_only(args):
    """Tree decode attention on a prebuilt tree (plan cached); K timed calls."""
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__ as g
    g.build()
    from copy_write_forked_gb300.runner import pool_for, run_script
    w, desc = other_workload(args.workload)
    pool = pool_for(w, extra_blocks=len(w.query) + 16, tc_min_rows=args.tc_min_rows,
                    fold_segments=args.fold_segments)   # room for one more token per queried branch
    h = run_script(pool, w, device=dev)
    br = [h[b] for b in w.query]
    Q = w.q(dev)
    out = torch.empty_like(Q)
    flush_r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    pool.sync()
    pool.tree_attn_decode(Q, br, out=out)        # builds the plan (and sizes the workspace)
    plan_first_us = pool.last_plan_stats()["plan_us"]
    rb = []
    Qr = Q.flip(0).contiguous()
    for _ in range(5):                           # rebuilds: another branch order misses the plan cache
        for qq, bb in ((Qr, br[::-1]), (Q, br)):
            pool.sync()                          # the device idle: time the planning alone
            pool.tree_attn_decode(qq, bb, out=out)
            rb.append(pool.last_plan_stats()["plan_us"])
    pool.sync()
    for _ in range(args.warmup):
        flush_r.max()
        pool.tree_attn_decode(Q, br, out=out)
    pool.set_profiling(True)
    part, tot, tcms = [], [], []
    for _ in range(args.steps):
        flush_r.max()
        pool.tree_attn_decode(Q, br, out=out)
        tm = pool.last_timings()
        part.append(tm["attn_partial"])
        tot.append(tm["attn_total"])
        if tm.get("attn_tc") is not None:
            tcms.append(tm["attn_tc"])
    pool.sync()
    st = pool.last_plan_stats()
    unique = w.unique_kv_bytes() + Q.numel() * Q.element_size()
    pk_ms, tot_ms = statistics.median(part), statistics.median(tot)
    # one more token on every queried branch, then the host side of the next
    # call: a refresh of the cached plan if no branch reached a new block
    # (after the timed calls, so they see the tree as described)
    g1 = torch.Generator(device=dev).manual_seed(1234)
    K1 = torch.randn((len(br), 1, w.n_kv_heads, w.head_dim), generator=g1, device=dev).to(w.dtype)
    pool.append_kv(br, K1, K1.clone())
    pool.sync()
    pool.tree_attn_decode(Q, br, out=out)
    st1 = pool.last_plan_stats()
    after_one = {"plan_us": st1["plan_us"], "refreshed": bool(st1["refreshed"])}
    pool.sync()
    peak, src = read_peaks()
    ach = unique / (pk_ms / 1e3) / 1e9
    nq = len(w.query) * w.q_len
    line = {"metric": "tree decode attn branch-queries/s & HBM GB/s (unique KV) vs peak; fork us",
            "workload": args.workload, "value": nq / (tot_ms / 1e3), "unit": "branch-queries/s",
            "ms_per_call": tot_ms, "partial_kernel_ms": pk_ms,
            "p10_p90_ms": {"call": [quantile(tot, 0.1), quantile(tot, 0.9)],
                           "partial_kernels": [quantile(part, 0.1), quantile(part, 0.9)]},
            "steps": args.steps, "warmup": args.warmup,
            "dtype": "bf16", "data": "synthetic (Q/K/V ~ N(0,1), seeded)",
            "config": {"workload": desc, "step": "tree decode attention on a prebuilt tree (plan cached)",
                       "l2": "flushed between calls (256 MiB read)"},
            "tc_kernel_ms": statistics.median(tcms) if tcms else None,
            "host_plan_us": {"first_call": plan_first_us, "rebuild_median": statistics.median(rb),
                             "after_one_more_token": after_one},
            "roofline": {"bound": "hbm",
                         "kernel": ("k_attn_partial_tc + " if st["n_tc_units"] else "") + "k_attn_partial_bf16",
                         "achieved": ach, "peak": peak,
                         "peak_source": src, "unit": "GB/s", "frac": ach / peak, "algorithmic_bytes": unique},
            "plan": st}
    print(json.dumps(line), flush=True)
    pool.close()


def fork_latency(dev, reps=200):
    """Fork of a chain of `depth` blocks whose tail block is half full, with 1
    and 4 children (then freed).  Three views per call: the host time of the C
    call, the device time between events recorded around the launch, and the
    round trip (call + stream synchronisation)."""
    import ctypes
    import torch
    from copy_write_forked_gb300.dendrite import Pool, lib
    L = lib()
    res = {}
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    for depth in (1, 10, 50, 100, 500):
        n = depth * 16 - 8
        pool = Pool(depth + 64, 16, 8, 128, torch.bfloat16, max_branches=16, max_blocks_per_branch=depth + 4)
        r = pool.new_branch()
        K = torch.zeros(1, n, 8, 128, dtype=torch.bfloat16, device=dev)
        pool.append_kv([r], K, K)
        pool.sync()
        for nc in (1, 4):
            out = (ctypes.c_int32 * nc)()
            host, gpu, rt = [], [], []
            for i in range(reps):
                pool.set_profiling(i % 2 == 1)
                stream.synchronize()
                t0 = time.perf_counter()
                rc = L.dendrite_fork(pool._h, r, nc, out, sp)
                t1 = time.perf_counter()
                stream.synchronize()
                t2 = time.perf_counter()
                assert rc == 0
                if i % 2 == 1:
                    gpu.append(pool.last_timings()["fork"] * 1e3)
                else:
                    host.append((t1 - t0) * 1e6)
                    rt.append((t2 - t0) * 1e6)
                pool.free(list(out))
            res[f"depth{depth}_children{nc}"] = {
                "host_call_us": statistics.median(host[5:]),
                "gpu_event_us": statistics.median(gpu[5:]),
                "round_trip_us": statistics.median(rt[5:])}
        pool.close()
    return res


# ------------------------------------------------------------ oracle arm
def _oracle_sample(seconds: float):
    """Runs in a fresh single-threaded process: the oracle's tree attention on
    branches of the beam workload until `seconds` of CPU work are spent."""
    import torch
    torch.set_num_threads(1)
    from copy_write_forked_gb300 import workloads as W
    from oracle import KVTree
    w = beam_workload(seed=0)
    ids = list(w.query[:4])                 # the 4 branches of request 0
    tree = _oracle_request_tree(w, 0)
    Q = [w.q_one(i) for i in range(4)]
    n = 0
    t0 = time.perf_counter()
    while True:
        tree.attend(ids[n % 4], Q[n % 4])
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return n, dt


def _oracle_request_tree(w, req):
    from oracle import KVTree
    pre = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == w.meta["prefix"])
    div = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == w.meta["divergent"])
    width = w.meta["width"]
    tree = KVTree(w.n_kv_heads, w.head_dim)
    tree.new_root(req)
    k, v = w.kv_one(pre, req)
    tree.append(req, k, v)
    kids = [w.query[req * width + j] for j in range(width)]
    tree.fork(req, kids)
    for j, c in enumerate(kids):
        k, v = w.kv_one(div, req * width + j)
        tree.append(c, k, v)
    return tree


def cpu_baseline(seconds: float):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, json; sys.path.insert(0, %r); import bench; n, dt = bench._oracle_sample(%f); "
            "print(json.dumps([n, dt]))" % (ROOT, seconds))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr[-300:]}
    n, dt = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": n / dt, "unit": "branch-queries/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} branch queries (fp64 tree attention, 4352-token branches of request 0 of the "
                      f"beam workload) in {dt:.1f} s, single thread"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    torch.set_num_threads(1)
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    from copy_write_forked_gb300 import workloads as W
    w = beam_workload(seed=0)
    tree = _oracle_request_tree(w, 0)
    ids = list(w.query[:4])
    Q = [w.q_one(i) for i in range(4)]

    k = [0]

    def step():
        # one branch query (round robin over the 4 branches of request 0)
        j = k[0] % 4
        tree.attend(ids[j], Q[j])
        k[0] += 1

    for _ in range(args.warmup):
        step()
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        t.append(time.perf_counter() - t0)
    ms = statistics.mean(t) * 1e3
    value = 1 / (ms / 1e3)
    line = {"impl": "reference",
            "metric": "tree decode attn branch-queries/s & HBM GB/s (unique KV) vs peak; fork us",
            "value": value, "unit": "branch-queries/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (Q/K/V ~ N(0,1), seeded)",
            "config": dict(config_of(w), parallelism="single thread"),
            "cpu_baseline": {"value": value, "unit": "branch-queries/s", "cores": 1, "kind": "oracle",
                             "sample": "per step: fp64 tree attention (materialise + softmax(qK^T/sqrt(d))V, "
                                       "32 heads) of one 4352-token branch of request 0, single thread"},
            "e2e": {"value": value, "unit": "branch-queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tc-min-rows", type=int, default=0,
                    help="segments with more query rows per KV head use the tcgen05 kernel (0: default 64, -1: off)")
    ap.add_argument("--fold-segments", type=int, default=0,
                    help="fold short shared segments into the ones that follow (0: default, k: below k percent "
                         "of the estimate, -1: off)")
    ap.add_argument("--workload", default="beam", choices=["beam", "mcts", "specverify", "stress", "decode32"],
                    help="beam = the full-path step (default JSON line); others time tree attention only")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "ours" and args.workload == "decode32":
        run_decode_layers(args)
        return
    if args.impl == "ours" and args.workload != "beam":
        run_attention_only(args)
        return
    if args.impl == "reference":
        # the oracle runs single-threaded: pin BLAS/OpenMP pools before numpy loads
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
