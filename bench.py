#!/usr/bin/env python3
"""Benchmark of the copy-on-write tree KV cache hot path on GB300.

Workload (default, ``--workload stress``): Llama-3-8B-shaped attention layer
(32 Q heads, 8 KV heads, head_dim 128, bf16, block_size 16); 16 independent
requests with a 32768-token shared prefix, forked 64 ways, each branch 1024
divergent tokens, one decode query per branch (1024 branch queries).  The
prefixes are prefilled once before timing (resident in HBM).  One step is one
pass of the whole path over that batch:

    fork (16 parents x 64 children, batched)  ->  copy-on-write append of the
    1024 divergent tokens of all 1024 branches  ->  tree decode attention
    (plan, shared-prefix + leaf partials, log-sum-exp merge)  ->  free of the
    1024 branches

``--workload beam`` runs the same step on 8 requests x 4096-token prefix,
fork 4, 256 divergent tokens.  ``mcts``, ``specverify`` and ``stressattn`` time
tree attention alone on a prebuilt tree; ``decode32`` runs the beam step
through 32 layers; ``forks`` times the 100,000 batched forks of the stress
configuration alone.

`value` is branch-queries per second of step time (all ranks summed).  The
``roofline`` entry covers the kernel that takes the most time in the step,
with its algorithmic bytes over its CUDA-event duration; ``roofline_attention``
covers the attention partial kernels against the unique KV bytes (each shared
block counted once) plus Q.

`--impl reference` times the fp64 CPU oracle on the host cores: every step,
one worker process per core runs the oracle's tree attention of one branch of
the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
W_SEED_DECODE = 4242          # seed of the decode step's new K/V rows
METRIC = "tree decode attn branch-queries/s & HBM GB/s (unique KV) vs peak; fork us"


# ------------------------------------------------------------------ helpers

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


# Kernel -> source file, for matching a recorded ncu capture to the code it was taken on.
KERNEL_SOURCES = {
    "k_append_copy": "copy_write_forked_gb300/csrc/pool.cu",
    "k_attn_partial_tc": "copy_write_forked_gb300/csrc/attn_tc.cu",
    "k_attn_partial_bf16": "copy_write_forked_gb300/csrc/attn.cu",
}


def source_sha(kernel: str) -> str:
    with open(os.path.join(ROOT, KERNEL_SOURCES[kernel]), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of ``kernel`` on ``workload`` from
    the ncu table in profiles/ncu_traffic.md, if it was taken on the current
    source of that kernel's file; None otherwise (no capture, or the kernel's
    source changed since)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    if " + " in kernel:   # kernels timed together: the sum of their own captures
        parts = [recorded_traffic(k, workload) for k in kernel.split(" + ")]
        return None if any(x is None for x in parts) else sum(parts)
    sha = source_sha(kernel)
    for line in open(path):
        f = [x.strip() for x in line.strip().strip("|").split("|")]
        if len(f) >= 7 and f[0] == kernel and f[1] == workload and f[2] == sha:
            try:
                return int(f[6].replace(",", ""))
            except ValueError:
                return None
    return None


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


# ------------------------------------------------------------ workloads
FULL_PATH = {
    # name: (requests, prefix, fork width, divergent tokens, description)
    "stress": (16, 32768, 64, 1024, "large fork + CoW stress, Llama-3-8B attention layer: 16 requests x "
                                    "32768-token prefix, fork 64, 1024 divergent tokens per branch"),
    "beam": (8, 4096, 4, 256, "beam-like 4-way fork, Llama-3-8B attention layer: 8 requests x 4096-token "
                              "prefix, fork 4, 256 divergent tokens per branch"),
}


def full_path_workload(name: str, seed: int = 0, requests=None):
    from copy_write_forked_gb300 import workloads as W
    R, P, Wd, Dv, _ = FULL_PATH[name]
    w = W.beam(requests=requests or R, prefix=P, width=Wd, divergent=Dv, seed=seed)
    if name == "stress":
        w.name = f"stress_r{requests or R}_p{P}_w{Wd}_div{Dv}"
    return w


def config_of(w, name):
    m = w.meta
    big = w.unique_kv_bytes() > (256 << 20)
    return {"workload": FULL_PATH[name][4] if m["requests"] == FULL_PATH[name][0] else
            FULL_PATH[name][4] + f" (reduced to {m['requests']} requests)",
            "name": w.name, "requests": m["requests"], "prefix_tokens": m["prefix"], "fork_width": m["width"],
            "divergent_tokens": m["divergent"], "branch_queries_per_step": len(w.query),
            "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size,
            "l2": ("not flushed: inputs larger than L2 (%.1f GB of unique KV read and %.1f GB of new rows "
                   "written per step)" % (w.unique_kv_bytes() / 1e9, _divergent_bytes(w) / 1e9)) if big else
                  "flushed before every step (read-only pass over 256 MiB)",
            "step": "fork + CoW append of the divergent tokens + tree decode attention + free "
                    "(the tree below each fork is rebuilt by every step; the prefixes stay resident)"}


def _divergent_bytes(w):
    m = w.meta
    return 2 * len(w.query) * m["divergent"] * w.n_kv_heads * w.head_dim * 2


# ---------------------------------------------------------- our arm
def _step_desc(kind):
    if kind == "decode":
        return ("decode step on the prebuilt tree: every leaf forks one child (batched fork), each child "
                "appends one new token (copy-on-write of the leaf's partially filled tail block), tree decode "
                "attention for the children, free of the old leaves (the children are the next step's leaves; "
                "each step adds one token per branch)")
    return ("fork of the prefixes + CoW append of all divergent tokens + tree decode attention + free (the tree "
            "below each fork is rebuilt by every step; the prefixes stay resident)")


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

    name, kind = args.workload, args.step
    w = full_path_workload(name, seed=rank, requests=args.requests)
    R, P, Wd, Dv = (w.meta[k] for k in ("requests", "prefix", "width", "divergent"))
    nq, nkv, d = w.n_q_heads, w.n_kv_heads, w.head_dim
    bs = w.block_size
    nl = R * Wd                                   # branches queried per step
    n_prof = min(args.steps, 100 if name == "beam" else 20)
    e2e_steps = args.steps if name == "beam" else min(args.steps, 50)
    # decode steps the run takes in all (warm-up, timed, profiled twice, e2e
    # warm-up and timed, the checked step)
    total_steps = args.warmup + args.steps + 2 * n_prof + 2 * args.warmup + e2e_steps + 2
    grow = total_steps if kind == "decode" else 0
    nblocks = R * (P // bs + 1) + nl * (Dv // bs + 3 + grow // bs) + 64
    from copy_write_forked_gb300 import workloads as W
    pool = Pool(nblocks, bs, nkv, d, torch.bfloat16, max_branches=R + 2 * nl + 16,
                max_blocks_per_branch=(P + Dv + grow) // bs + 8,
                turbo=W.turbo_codec(rank) if args.turbo else None, device_planning=args.device_planning,
                tc_sms=args.tc_sms, pack_segments=args.pack_segments)
    # prefill (untimed): the prefixes, resident in HBM
    roots = [pool.new_branch() for _ in range(R)]
    prefill_idx = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == P)
    Kp, Vp = w.kv(prefill_idx, dev)
    pool.append_kv(roots, Kp, Vp)
    pool.sync()
    del Kp, Vp
    div_idx = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == Dv)
    Kd, Vd = w.kv(div_idx, dev)            # divergent tokens of all branches
    Q = w.q(dev)
    out = torch.empty_like(Q)
    stream = torch.cuda.current_stream()
    state = {"leaves": None, "s": 0}
    if kind == "decode":
        # the tree of the configuration, built once: fork, divergent tokens
        kids = pool.fork_batch(roots, [Wd] * R)
        state["leaves"] = [c for ks in kids for c in ks]
        pool.append_kv(state["leaves"], Kd, Vd)
        pool.sync()
        del Kd, Vd
        gen = torch.Generator(device=dev).manual_seed(W_SEED_DECODE + rank)
        Kn = torch.randn((nl, 1, nkv, d), generator=gen, device=dev).to(torch.bfloat16)
        Vn = torch.randn((nl, 1, nkv, d), generator=gen, device=dev).to(torch.bfloat16)
    else:
        Kn, Vn = Kd, Vd
    pool.sync()
    big = w.unique_kv_bytes() > (256 << 20)
    flush_r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        # read-only pass over 256 MiB (2x L2): evicts the cache and leaves it
        # holding clean lines, so no write-back lands inside the next step.
        # Workloads whose inputs are far larger than L2 skip it.
        if not big:
            flush_r.max()

    def step(K=None, V=None, Qs=None, o=None, check=None):
        K = Kn if K is None else K
        V = Vn if V is None else V
        Qs = Q if Qs is None else Qs
        o = out if o is None else o
        if kind == "decode":
            br = pool.fork_each(state["leaves"])
            pool.append_kv(br, K, V)
            pool.tree_attn_decode(Qs, br, out=o)
            if check is not None:
                # the same call again on the same tree (before the parents
                # are freed, which may regroup the tree's segments): the
                # cached plan and the same kernels give the same bits
                pool.tree_attn_decode(Q, br, out=check)
            pool.free(state["leaves"])
            state["leaves"] = br
            state["s"] += 1
        else:
            kids = pool.fork_batch(roots, [Wd] * R)
            br = [c for ks in kids for c in ks]
            pool.append_kv(br, K, V)
            pool.tree_attn_decode(Qs, br, out=o)
            pool.free(br)
        return br

    def rewind(s_to):
        # Untimed: roll every branch back to its length after decode step
        # s_to (truncate).  Each decode step adds one token to every branch,
        # so the passes after the timed one (per-kernel events, end to end)
        # would otherwise read a larger tree per step than the timed steps
        # did; rewound, they repeat the timed steps' tree sizes.
        if kind != "decode" or state["s"] == s_to:
            return
        if pool.branch_len(state["leaves"][0]) != P + Dv + state["s"]:
            raise RuntimeError("unexpected branch length")
        pool.truncate(state["leaves"], [P + Dv + s_to] * len(state["leaves"]))
        state["s"] = s_to

    def unique_tokens():
        # tokens the next step's queries see, each shared one once
        extra = state["s"] + 1 if kind == "decode" else 0
        return R * P + nl * (Dv + extra)

    # K + V bytes of one token in the pool (the records of a compressed pool)
    kv_tok = nkv * (96 + 64) if args.turbo else 2 * nkv * d * 2
    clk = ClockSampler(local).__enter__()
    pool.set_profiling(False)
    for _ in range(args.warmup):
        flush_l2()
        step()
    pool.sync()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    s_timed0 = state["s"]
    # ---- timed region: K steps enqueued back to back, one event pair per step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    tok_timed = []
    t_clk0 = time.time()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        tok_timed.append(unique_tokens())
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
    value = world * nl / (ms / 1e3)
    ref_out = out.clone()

    # ---- per-kernel device times (profiling events inside the library; one
    # synchronised step at a time so the events of each call can be read)
    pool.set_profiling(True)
    kern = {k: [] for k in ("fork", "append_meta", "append_copy", "attn_partial", "attn_tc", "attn_mma_side",
                            "attn_merge", "free", "attn_total")}
    plan_us, tok_prof = [], []
    orig_attn = pool.tree_attn_decode

    def attn_after_flush(*a, **k):
        # A read pass sits right before the attention call: the device works
        # through it while the host builds the plan and launches, so the
        # events around the attention kernels time the kernels, not the host.
        flush_r.max()
        return orig_attn(*a, **k)

    pool.tree_attn_decode = attn_after_flush
    rewind(s_timed0)
    for i in range(n_prof):
        flush_l2()
        tok_prof.append(unique_tokens())
        step()
        tm = pool.last_timings()
        plan_us.append(pool.last_plan_stats()["plan_us"])
        for k in kern:
            if tm.get(k) is not None:
                kern[k].append(tm[k])
    # the same steps with events around whole attention calls only: the
    # call's kernels then overlap one another as they do unprofiled
    pool.set_profiling(2)
    call_light, tok_light = [], []
    rewind(s_timed0)
    for i in range(n_prof):
        flush_l2()
        tok_light.append(unique_tokens())
        step()
        call_light.append(pool.last_timings()["attn_total"])
    pool.tree_attn_decode = orig_attn
    pool.set_profiling(False)
    km = {k: (statistics.mean(v) if v else None) for k, v in kern.items()}

    peak, peak_src = read_peaks()
    plan = pool.last_plan_stats()
    q_bytes = Q.numel() * Q.element_size()
    uniq = statistics.mean(tok_prof) * kv_tok
    # algorithmic bytes per launch of each of the step's large kernels
    append_bytes = 2 * (Kn.numel() + Vn.numel()) * Kn.element_size()     # rows read once and written once
    tc_ms = km["attn_tc"] or 0.0
    # the mma.sync kernel runs beside the tcgen05 one when both have work; it
    # then has its own events (on the library's side stream)
    mma_ms = km["attn_mma_side"] if km.get("attn_mma_side") else km["attn_partial"] - tc_ms
    prefix_bytes = R * P * kv_tok                     # shared prefixes: the tcgen05 class when it exists
    cand = {"k_append_copy": (km["append_copy"], append_bytes, "new K and V rows read once and written once")}
    concurrent = bool(km.get("attn_mma_side")) and bool(tc_ms)
    if concurrent:
        # the two partial kernels run side by side on the HBM: they are timed,
        # and bound, together (each one's own span includes the other's share)
        cand["k_attn_partial_tc + k_attn_partial_bf16"] = (
            km["attn_partial"], uniq + q_bytes,
            "unique KV (each shared block once) + Q, both partial kernels running concurrently")
    elif tc_ms:
        cand["k_attn_partial_tc"] = (tc_ms, prefix_bytes + q_bytes,
                                     "unique KV of the shared prefixes (each block once) + Q")
        cand["k_attn_partial_bf16"] = (mma_ms, uniq - prefix_bytes + q_bytes,
                                       "unique KV of the branches' own blocks + Q")
    else:
        cand["k_attn_partial_bf16"] = (mma_ms, uniq + q_bytes, "unique KV (each shared block once) + Q")
    dom = max(cand, key=lambda k: cand[k][0])

    def roof(kernel, kms, nbytes, what, traffic):
        ach = nbytes / (kms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": kernel, "achieved": ach, "peak": peak, "peak_source": peak_src,
                "unit": "GB/s", "frac": ach / peak, "traffic": traffic,
                "algorithmic_bytes": nbytes, "bytes_counted": what, "kernel_ms": kms}

    traffic_key = w.name + ("" if kind == "divergent" else "_decode")
    roofline = roof(dom, *cand[dom], recorded_traffic(dom, traffic_key))
    attn_roof = roof(("k_attn_partial_tc + " if tc_ms else "") + "k_attn_partial_bf16", km["attn_partial"],
                     uniq + q_bytes, "unique KV (each shared block once) + Q", None)
    attn_roof["per_kernel"] = {k: roof(k, *cand[k], recorded_traffic(k, traffic_key))
                               for k in cand if k.startswith("k_attn")}
    if concurrent:
        attn_roof["concurrent_kernel_ms"] = {"k_attn_partial_tc": tc_ms, "k_attn_partial_bf16": mma_ms,
                                             "note": "each kernel's span while sharing the GPU with the other"}
    # the call: plan upload (and expansion), partial kernels, merge, timed
    # with events around the whole call only
    call_ms = statistics.mean(call_light)
    uniq_light = statistics.mean(tok_light) * kv_tok
    attn_roof["call_ms"] = call_ms
    attn_roof["call_frac"] = (uniq_light + q_bytes) / (call_ms / 1e3) / 1e9 / peak
    attn_roof["call_ms_with_per_kernel_events"] = km["attn_total"]

    # ----- e2e through the public API with host buffers (pinned), H2D + D2H inside
    # the timed region.  A copy stream brings step i + 1's K, V and Q in while
    # the compute stream runs step i (two device buffer sets); the result of
    # every step is read back to pinned host memory on the compute stream.
    Kh = torch.empty(Kn.shape, dtype=Kn.dtype, pin_memory=True)
    Vh = torch.empty(Vn.shape, dtype=Vn.dtype, pin_memory=True)
    Qh = torch.empty(Q.shape, dtype=Q.dtype, pin_memory=True)
    Kh.copy_(Kn)
    Vh.copy_(Vn)
    Qh.copy_(Q)
    if kind == "divergent":
        del Kd, Vd
    Kn = Vn = None
    outh = [torch.empty(Q.shape, dtype=Q.dtype, pin_memory=True) for _ in range(2)]
    bufs = [(torch.empty(Kh.shape, dtype=Kh.dtype, device=dev), torch.empty(Vh.shape, dtype=Vh.dtype, device=dev),
             torch.empty_like(Q), torch.empty_like(Q)) for _ in range(2)]
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

    ev_done = [torch.cuda.Event() for _ in range(2)]   # step using buffer set j computed its output

    def e2e_step(j, check=None):
        K2, V2, Q2, o2 = bufs[j]
        stream.wait_event(ev_in[j])
        br = step(K2, V2, Q2, o2, check=check)
        # the result goes back on the copy stream, beside the next step
        ev_done[j].record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_done[j])
            outh[j].copy_(o2, non_blocking=True)
            ev_used[j].record(copy_stream)
        return br

    def e2e_run(n, check=None):
        bring_in(0)
        br = None
        for i in range(n):
            if i + 1 < n:
                bring_in((i + 1) % 2)
            br = e2e_step(i % 2, check=check if i == n - 1 else None)
        return br

    # the e2e warm-up steps end where the timed steps began (a branch keeps
    # at least one divergent token)
    rewind(max(s_timed0 - 2 * args.warmup, 1 - Dv))
    for _ in range(args.warmup):
        flush_l2()
        e2e_run(2)
    torch.cuda.synchronize()
    tok_e2e = [unique_tokens() + (nl * i if kind == "decode" else 0) for i in range(e2e_steps)]
    flush_l2()
    torch.cuda.synchronize()
    e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    e2e_ev[0].record(stream)
    copy_stream.wait_stream(stream)
    e2e_run(e2e_steps)
    stream.wait_stream(copy_stream)
    e2e_ev[1].record(stream)
    torch.cuda.synchronize()
    e2e = max_over_ranks(e2e_ev[0].elapsed_time(e2e_ev[1]) / e2e_steps, world, dev)
    # one more (untimed) e2e step whose attention is repeated on the device
    # for the bit-exact check below
    chk = torch.empty_like(Q)
    e2e_run(1, check=chk if kind == "decode" else None)
    torch.cuda.synchronize()
    h2d = (Kh.numel() + Vh.numel() + Qh.numel()) * 2
    d2h = outh[0].numel() * 2
    # The last e2e step's output equals, bit for bit, the device-resident
    # attention of the same queries over the same tree (same plan, same kernels).
    if kind != "decode":
        chk = ref_out         # every divergent step rebuilds the same tree
    torch.cuda.synchronize()
    if not torch.equal(outh[0].to(dev), chk):
        raise RuntimeError("e2e output differs from the device-resident attention")
    pool.sync()
    pool.close()
    del bufs, Kh, Vh, outh
    torch.cuda.empty_cache()

    # ----- fork latency at depths 1..500 blocks (tail half full), 1 and 4 children,
    # and the 100,000 batched forks with copy-on-write appends of the stress configuration
    fork = fork_latency(dev) if rank == 0 else {}
    forks100k = fork_stress_timed(dev) if rank == 0 and not args.no_fork_stress else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds, name)

    # fork 1 + append 2 (meta, copy) + attention (a new tree needs a new plan:
    # its upload, the tcgen05 kernel when the plan has such units, the
    # mma.sync kernel, the merge) + free 1
    per_step = 1 + 2 + (4 if plan["n_tc_units"] else 3) + 1
    cfg = config_of(w, name)
    cfg["step"] = _step_desc(kind)
    if kind == "decode" and w.unique_kv_bytes() > (256 << 20):
        cfg["l2"] = ("not flushed: inputs larger than L2 (%.1f GB of unique KV read per step; each branch writes "
                     "one new token and copies its parent's partially filled tail block)"
                     % (statistics.mean(tok_timed) * kv_tok / 1e9))
    if args.turbo:
        cfg["kv_storage"] = ("compressed blocks (TurboQuant records: 96-byte keys, 64-byte values per token and "
                             "head, 3.2x smaller than bf16); algorithmic bytes count the records")
    if kind == "decode":
        # each branch's decoded tokens beyond the configuration's, first and last timed step
        cfg["decoded_tokens_per_branch_timed"] = [(tok_timed[0] - R * P) // nl - Dv - 1,
                                                  (tok_timed[-1] - R * P) // nl - Dv - 1]
    cfg["unique_kv_bytes_timed_mean"] = statistics.mean(tok_timed) * kv_tok
    line = {
        "metric": METRIC,
        "value": value, "unit": "branch-queries/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (Q/K/V ~ N(0,1), seeded)",
        "config": dict(cfg, parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                       planning={-1: "host", 0: "default (units and CTA split on the device for plans of "
                                                 "2048+ units averaging under 32 tiles per unit)",
                                 1: "units and CTA split on the device"}[args.device_planning]),
        "roofline": roofline,
        "roofline_attention": attn_roof,
        "cpu_baseline": cpu,
        "e2e": {"value": world * nl / (e2e / 1e3), "unit": "branch-queries/s", "ms_per_step": e2e,
                "unique_kv_bytes_mean": statistics.mean(tok_e2e) * kv_tok,
                "steps": e2e_steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": per_step * args.steps,
        "clocks": clocks,
        "kernels_ms": km,
        "attn_branch_queries_per_s": nl / (km["attn_total"] / 1e3),
        "plan": {"segments": plan["n_segments"], "units": plan["n_units"], "ctas": plan["n_ctas"],
                 "tc_units": plan["n_tc_units"], "tc_ctas": plan["n_tc_ctas"],
                 "partials": plan["n_partials"], "tiles": plan["tiles"], "unique_tiles": plan["unique_tiles"],
                 "host_plan_us_mean": statistics.mean(plan_us)},
        "fork_us": fork,
        "forks_100k": forks100k,
        "wall_s": wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
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
    w = full_path_workload("beam", seed=rank)
    R, P, Wd, Dv = (w.meta[k] for k in ("requests", "prefix", "width", "divergent"))
    nq, nkv, d, bs = w.n_q_heads, w.n_kv_heads, w.head_dim, w.block_size
    nblocks = R * (P // bs + 1) + R * Wd * (Dv // bs + 2) + 64
    pool = Pool(nblocks, bs, nkv, d, torch.bfloat16, max_branches=R * (Wd + 1) + 8,
                max_blocks_per_branch=(P + Dv) // bs + 8, n_layers=NL, device_planning=args.device_planning,
                pack_segments=args.pack_segments)
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
    layer_ms = {k: [] for k in ("append_copy", "attn_partial", "attn_merge", "attn_total")}
    for l in range(NL):
        pool.append_layer(l, Kd[l][0], Kd[l][1])
        flush_r.max()
        pool.tree_attn_decode(Q, br, out=outs[l], layer=l)
        tm = pool.last_timings()
        part.append(tm["attn_partial"])
        for k in layer_ms:
            if tm.get(k) is not None:
                layer_ms[k].append(tm[k])
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
            "per_layer_kernel_ms_median": {k: (statistics.median(v) if v else None) for k, v in layer_ms.items()},
            "per_layer_ms": step_ms / NL,
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
    if name == "stressattn":
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
    pool = pool_for(w, extra_blocks=len(w.query) + 16, tc_min_rows=args.tc_min_rows, tc_sms=args.tc_sms,
                    pack_segments=args.pack_segments,
                    fold_segments=args.fold_segments,   # room for one more token per queried branch
                    device_planning=args.device_planning)
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
    part, tot, tcms, mms = [], [], [], []
    for _ in range(args.steps):
        flush_r.max()
        pool.tree_attn_decode(Q, br, out=out)
        tm = pool.last_timings()
        part.append(tm["attn_partial"])
        tot.append(tm["attn_total"])
        if tm.get("attn_tc") is not None:
            tcms.append(tm["attn_tc"])
        if tm.get("attn_mma_side") is not None:
            mms.append(tm["attn_mma_side"])
    pool.sync()
    # whole calls only (their kernels overlap as they do unprofiled)
    pool.set_profiling(2)
    tot_light = []
    for _ in range(args.steps):
        flush_r.max()
        pool.tree_attn_decode(Q, br, out=out)
        tot_light.append(pool.last_timings()["attn_total"])
    pool.set_profiling(False)
    pool.sync()
    st = pool.last_plan_stats()
    unique = w.unique_kv_bytes() + Q.numel() * Q.element_size()
    pk_ms, tot_ms = statistics.median(part), statistics.median(tot_light)
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
            "ms_per_call_with_per_kernel_events": statistics.median(tot),
            "p10_p90_ms": {"call": [quantile(tot_light, 0.1), quantile(tot_light, 0.9)],
                           "partial_kernels": [quantile(part, 0.1), quantile(part, 0.9)]},
            "steps": args.steps, "warmup": args.warmup,
            "dtype": "bf16", "data": "synthetic (Q/K/V ~ N(0,1), seeded)",
            "config": {"workload": desc, "step": "tree decode attention on a prebuilt tree (plan cached)",
                       "l2": "flushed between calls (256 MiB read)"},
            "tc_kernel_ms": statistics.median(tcms) if tcms else None,
            "mma_kernel_ms_beside_tc": statistics.median(mms) if mms else None,
            "host_plan_us": {"first_call": plan_first_us, "rebuild_median": statistics.median(rb),
                             "after_one_more_token": after_one},
            "roofline": {"bound": "hbm",
                         "kernel": ("k_attn_partial_tc + " if st["n_tc_units"] else "") + "k_attn_partial_bf16",
                         "achieved": ach, "peak": peak,
                         "peak_source": src, "unit": "GB/s", "frac": ach / peak, "algorithmic_bytes": unique},
            "plan": st}
    print(json.dumps(line), flush=True)
    pool.close()


def run_mcts_loop(args):
    """The MCTS demo's loop as a decode loop: root prompt of 2048 tokens; each
    iteration forks a uniformly chosen live leaf of depth < 12 into 4
    children, appends 32 tokens to each, and runs tree decode attention for
    every live leaf (a new query set, so a new plan, every iteration).  Per
    iteration: the host time of planning (inside the attention call), the
    attention call's device time, and the wall time of the iteration's three
    calls up to the attention's completion."""
    import torch
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__ as g
    g.build()
    from copy_write_forked_gb300 import workloads as W
    from copy_write_forked_gb300.runner import pool_for
    w = W.mcts(iters=args.mcts_iters)
    pool = pool_for(w, fold_segments=args.fold_segments, device_planning=args.device_planning,
                    pack_segments=args.pack_segments)
    gen = torch.Generator(device=dev).manual_seed(77)
    maxq = len(w.query)
    Qall = torch.randn((maxq, 1, w.n_q_heads, w.head_dim), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty_like(Qall)
    h = {}
    live = []
    rows = []
    pool.set_profiling(True)
    ops = w.ops
    i = 0
    while i < len(ops):
        op = ops[i]
        if op.kind == "new":
            h[op.branches[0]] = pool.new_branch()
            live.append(op.branches[0])
        elif op.kind == "append":            # the root prompt
            K, V = w.kv(i, dev)
            pool.append_kv([h[b] for b in op.branches], K, V)
        else:                                # one iteration: fork, then the children's append
            nxt = ops[i + 1]
            K, V = w.kv(i + 1, dev)
            pool.sync()
            t0 = time.perf_counter()
            kids = pool.fork_batch([h[p] for p in op.branches], [len(c) for c in op.children])
            for ch, hs in zip(op.children, kids):
                h.update(zip(ch, hs))
            for p, ch in zip(op.branches, op.children):
                live.remove(p)
                live.extend(ch)
            pool.append_kv([h[b] for b in nxt.branches], K, V)
            q = sorted(live)
            n = len(q)
            pool.tree_attn_decode(Qall[:n], [h[b] for b in q], out=out[:n])
            pool.sync()
            t1 = time.perf_counter()
            tm = pool.last_timings()
            st = pool.last_plan_stats()
            rows.append({"leaves": n, "plan_us": st["plan_us"], "call_us": tm["attn_total"] * 1e3,
                         "wall_us": (t1 - t0) * 1e6})
            i += 1
        i += 1
    pool.set_profiling(False)
    pool.close()
    last = rows[-100:]
    line = {"metric": METRIC, "workload": "mctsloop",
            "config": {"workload": "MCTS loop: root 2048, %d iterations of fork 4 x 32 tokens, tree decode "
                                   "attention over every live leaf after each iteration" % args.mcts_iters,
                       "timing": "per iteration, host plan time inside the attention call; device time of the "
                                 "attention call (CUDA events); wall time of fork + append + attention up to "
                                 "completion"},
            "iterations": len(rows),
            "last100": {"leaves_mean": statistics.mean(r["leaves"] for r in last),
                        "host_plan_us_mean": statistics.mean(r["plan_us"] for r in last),
                        "gpu_call_us_mean": statistics.mean(r["call_us"] for r in last),
                        "wall_us_mean": statistics.mean(r["wall_us"] for r in last)},
            "all": {"host_plan_us_mean": statistics.mean(r["plan_us"] for r in rows),
                    "gpu_call_us_mean": statistics.mean(r["call_us"] for r in rows),
                    "plan_below_call_fraction": sum(r["plan_us"] < r["call_us"] for r in rows) / len(rows)},
            "host_plan_vs_gpu_call_last100": statistics.mean(r["plan_us"] for r in last) /
                                             statistics.mean(r["call_us"] for r in last)}
    print(json.dumps(line), flush=True)


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
            skip = min(5, len(host) // 2)      # the first calls warm up
            res[f"depth{depth}_children{nc}"] = {
                "host_call_us": statistics.median(host[skip:]),
                "gpu_event_us": statistics.median(gpu[skip:]),
                "round_trip_us": statistics.median(rt[skip:])}
        pool.close()
    return res


def fork_stress_timed(dev, batches=5000):
    """The 100,000 batched forks of the stress configuration: chains of 1, 10,
    50, 100 and 500 blocks with a half-full tail block; every batch forks each
    chain 4 ways in one call (20 forks), appends one token to every child (each
    copies its chain's shared half block) and frees the children.  Timed with
    CUDA events around all batches (the device work of 3 calls per batch)."""
    import torch
    from copy_write_forked_gb300 import workloads as W
    from copy_write_forked_gb300.dendrite import Pool
    depths = (1, 10, 50, 100, 500)
    N = sum(depths) + len(depths) + 64
    pool = Pool(N, 16, 8, 128, torch.bfloat16, max_branches=64, max_blocks_per_branch=512)
    roots = []
    for d in depths:
        r = pool.new_branch()
        roots.append(r)
        L = W.fork_chain_script(d)
        K = torch.randn(1, L, 8, 128, device=dev).bfloat16()
        pool.append_kv([r], K, K)
    Kt = torch.randn(4 * len(roots), 1, 8, 128, device=dev).bfloat16()
    stream = torch.cuda.current_stream()

    def batch():
        kids = pool.fork_batch(roots, [4] * len(roots))
        flat = [c for ks in kids for c in ks]
        pool.append_kv(flat, Kt, Kt)
        pool.free(flat)
        return len(flat)

    for _ in range(50):
        batch()
    pool.sync()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    forks = sum(batch() for _ in range(batches))
    e1.record(stream)
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    t2 = time.perf_counter()
    dev_ms = e0.elapsed_time(e1)
    pool.sync()
    pool.close()
    return {"forks": forks, "batches": batches, "depths_blocks": list(depths), "children_per_chain": 4,
            "device_ms": dev_ms, "wall_ms": (t2 - t0) * 1e3, "host_issue_ms": (t1 - t0) * 1e3,
            "us_per_fork_device": dev_ms * 1e3 / forks, "us_per_batch_device": dev_ms * 1e3 / batches,
            "forks_per_s_device": forks / (dev_ms / 1e3),
            "per_batch": "fork_batch (5 chains x 4 children) + append of 1 token to 20 children "
                         "(each copies a 32 KiB shared half block) + free of the 20 children"}


# ------------------------------------------------------------ oracle arm
# The oracle runs in worker processes of their own (fresh interpreters, one
# thread each), one per host core used: each rebuilds the ancestor chain of
# one branch of the workload in the oracle's logical tree, then answers
# "step" (one fp64 tree attention of its branch) and "run <seconds>" (as many
# as fit) commands on stdin.

def _oracle_branch_tree(w, req, child):
    """The oracle's tree of one request, holding only the queried child's own rows."""
    from oracle import KVTree
    pre = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == w.meta["prefix"])
    div = next(i for i, op in enumerate(w.ops) if op.kind == "append" and op.n_new == w.meta["divergent"])
    width = w.meta["width"]
    tree = KVTree(w.n_kv_heads, w.head_dim)
    tree.new_root(req)
    k, v = w.kv_one(pre, req)
    tree.append(req, k, v)
    qi = req * width + child
    bid = w.query[qi]
    tree.fork(req, [bid])
    k, v = w.kv_one(div, qi)
    tree.append(bid, k, v)
    return tree, bid, w.q_one(qi)


def _oracle_worker(name, index):
    import torch
    torch.set_num_threads(1)
    w = full_path_workload(name, seed=0)
    R, width = w.meta["requests"], w.meta["width"]
    tree, bid, q = _oracle_branch_tree(w, index % R, (index // R) % width)
    tree.attend(bid, q)
    print("ready", flush=True)
    for line in sys.stdin:
        cmd = line.split()
        if not cmd or cmd[0] == "quit":
            break
        if cmd[0] == "step":
            t0 = time.perf_counter()
            tree.attend(bid, q)
            print(json.dumps(time.perf_counter() - t0), flush=True)
        elif cmd[0] == "run":
            secs, n = float(cmd[1]), 0
            t0 = time.perf_counter()
            while True:
                tree.attend(bid, q)
                n += 1
                if time.perf_counter() - t0 >= secs:
                    break
            print(json.dumps([n, time.perf_counter() - t0]), flush=True)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _mem_available_bytes():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


class OracleWorkers:
    """n single-threaded oracle processes, each holding one branch's chain."""

    PER_WORKER_BYTES = {"stress": 3 << 30, "beam": 1 << 29}

    def __init__(self, name, n):
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        env.pop("CUDA_VISIBLE_DEVICES", None)
        code = "import sys; sys.path.insert(0, %r); import bench; bench._oracle_worker(%r, %%d)" % (ROOT, name)
        self.procs = [subprocess.Popen([sys.executable, "-c", code % i], stdin=subprocess.PIPE,
                                       stdout=subprocess.PIPE, text=True, env=env) for i in range(n)]
        for p in self.procs:
            if p.stdout.readline().strip() != "ready":
                self.close()
                raise RuntimeError("oracle worker failed to start")

    @classmethod
    def fit(cls, name, want):
        """How many workers the host's cores and available memory allow."""
        n = max(1, min(want, host_cores()))
        avail = _mem_available_bytes()
        if avail:
            n = max(1, min(n, int(avail * 0.6) // cls.PER_WORKER_BYTES[name]))
        return n

    def _all(self, cmd):
        for p in self.procs:
            p.stdin.write(cmd + "\n")
            p.stdin.flush()
        return [json.loads(p.stdout.readline()) for p in self.procs]

    def step(self):
        return self._all("step")

    def run(self, seconds):
        return self._all("run %f" % seconds)

    def close(self):
        for p in self.procs:
            try:
                p.stdin.write("quit\n")
                p.stdin.flush()
            except Exception:
                pass
        for p in self.procs:
            try:
                p.wait(timeout=30)
            except Exception:
                p.kill()


def _branch_tokens(name):
    R, P, Wd, Dv, _ = FULL_PATH[name]
    return P + Dv


def cpu_baseline(seconds: float, name: str):
    """The oracle as it stands on a bounded sample of the workload: fp64 tree
    attention of single branches for about ``seconds`` per leg, first on one
    core, then on every host core (one worker per core, each on its own
    branch).  The all-cores figure is the reported value."""
    res = {}
    for leg, want in (("single", 1), ("all", host_cores())):
        n = OracleWorkers.fit(name, want)
        pool = OracleWorkers(name, n)
        try:
            out = pool.run(seconds)
        finally:
            pool.close()
        q = sum(c for c, _ in out)
        dt = max(t for _, t in out)
        res[leg] = {"value": q / dt, "cores": n, "queries": q, "seconds": dt}
    a, s1 = res["all"], res["single"]
    tok = _branch_tokens(name)
    return {"value": a["value"], "unit": "branch-queries/s", "cores": a["cores"], "kind": "oracle",
            "host_cores": host_cores(),
            "sample": f"{a['queries']} branch queries in {a['seconds']:.1f} s on {a['cores']} worker processes "
                      f"(one thread each, each on its own {tok}-token branch of the {name} workload; fp64 "
                      f"materialise + softmax(qK^T/sqrt(d))V over 32 heads)",
            "single_thread": {"value": s1["value"], "cores": 1,
                              "sample": f"{s1['queries']} branch queries in {s1['seconds']:.1f} s, one thread"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    name = args.workload if args.workload in FULL_PATH else "stress"
    w = full_path_workload(name, seed=0)
    n = OracleWorkers.fit(name, host_cores())
    pool = OracleWorkers(name, n)
    try:
        for _ in range(args.warmup):
            pool.step()
        t = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            pool.step()
            t.append(time.perf_counter() - t0)
    finally:
        pool.close()
    ms = statistics.mean(t) * 1e3
    value = n / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC,
            "value": value, "unit": "branch-queries/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (Q/K/V ~ N(0,1), seeded)",
            "config": dict(config_of(w, name), parallelism=f"{n} host worker processes"),
            "cpu_baseline": {"value": value, "unit": "branch-queries/s", "cores": n, "kind": "oracle",
                             "sample": f"per step: {n} fp64 tree attentions (materialise + softmax(qK^T/sqrt(d))V, "
                                       f"32 heads), one per worker process, each on its own "
                                       f"{_branch_tokens(name)}-token branch of the {name} workload"},
            "e2e": {"value": value, "unit": "branch-queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_forks(args):
    """The 100,000 batched forks alone, plus fork latency by depth."""
    import torch
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__ as g
    g.build()
    line = {"metric": METRIC, "workload": "forks", "forks_100k": fork_stress_timed(dev, args.fork_batches),
            "fork_us": fork_latency(dev, args.fork_reps)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fork-stress", action="store_true")
    ap.add_argument("--fork-reps", type=int, default=200, help="--workload forks: calls per fork-latency point")
    ap.add_argument("--fork-batches", type=int, default=5000,
                    help="--workload forks: batches of the timed fork stress (20 forks each)")
    ap.add_argument("--turbo", action="store_true",
                    help="full-path workloads on a pool of compressed blocks (TurboQuant records)")
    ap.add_argument("--step", default="decode", choices=["decode", "divergent"],
                    help="full-path workloads: 'decode' (default) forks every leaf of the prebuilt tree once, "
                         "appends one token per child, attends and frees the old leaves; 'divergent' rebuilds "
                         "the tree below the prefixes (fork + append of all divergent tokens) every step")
    ap.add_argument("--mcts-iters", type=int, default=500, help="--workload mctsloop: iterations")
    ap.add_argument("--requests", type=int, default=None,
                    help="full-path workloads: fewer requests than the configuration (a smaller case for ncu)")
    ap.add_argument("--tc-min-rows", type=int, default=0,
                    help="segments with more query rows per KV head use the tcgen05 kernel (0: default 64, -1: off)")
    ap.add_argument("--pack-segments", type=int, default=0,
                    help="pack a segment's leaf followers into it as masked tiles (0: default, k: below k percent "
                         "of the estimate, -1: off)")
    ap.add_argument("--tc-sms", type=int, default=0,
                    help="SMs given to the tcgen05 kernel when both partial kernels have work (0: library "
                         "default, an estimate picks the split or none; -1: never split)")
    ap.add_argument("--device-planning", type=int, default=0, choices=[-1, 0, 1],
                    help="bf16 attention plans: expand units and the CTA split on the device (1), on the host (-1), "
                         "or by the library's default rule (0)")
    ap.add_argument("--fold-segments", type=int, default=0,
                    help="fold short shared segments into the ones that follow (0: default, k: below k percent "
                         "of the estimate, -1: off)")
    ap.add_argument("--workload", default="stress",
                    choices=["stress", "beam", "mcts", "specverify", "stressattn", "decode32", "forks", "mctsloop"],
                    help="stress (default) and beam: the full-path step; mcts, specverify, stressattn: tree "
                         "attention alone; decode32: the beam step through 32 layers; forks: the 100,000 "
                         "batched forks and fork latency; mctsloop: the MCTS demo's fork / append / attend "
                         "loop with host planning against the device call")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # the oracle runs single-threaded per worker: pin BLAS/OpenMP pools before numpy loads
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        run_reference(args)
    elif args.workload == "decode32":
        run_decode_layers(args)
    elif args.workload == "forks":
        run_forks(args)
    elif args.workload == "mctsloop":
        run_mcts_loop(args)
    elif args.workload in FULL_PATH:
        run_ours(args)
    else:
        run_attention_only(args)


if __name__ == "__main__":
    main()
