"""Seeded synthetic workloads for the copy-on-write KV tree.

This module only *describes* work: operation scripts (which branch is created,
forked, appended to, freed and queried) and the random Q/K/V values those
operations carry.  It holds none of the method's arithmetic (no attention, no
block allocation, no copy-on-write decision, no merge), so both the CUDA path
and the fp64 oracle can consume the very same inputs without sharing any
method code.

Branches are named by *logical ids* (0, 1, 2, ... in creation order).  Each
consumer maps logical ids to whatever handles its own implementation returns.

Workload shapes follow the pages' settings (Dendrite article, section
"技术深度解析": Llama 3 8B decoding with 4-way fork search and multi-draft
speculation; dendrite demo.tape, section "MCTS demo": 500 iterations,
branching factor 4, max depth 12, head_dim 128, 2048-token context).  All values
are synthetic: Q/K/V ~ N(0, 1) drawn from a seeded torch generator and rounded
to the pool dtype.  No dataset or model weights are involved.
"""
from __future__ import annotations

import hashlib
import random
from dataclasses import dataclass, field
from typing import Dict, List, Sequence, Tuple

import torch

__all__ = [
    "Op", "Workload", "seed_of",
    "tiny_cow", "beam", "mcts", "spec_verify", "fork_stress_attention",
    "fork_chain_script", "random_script", "turbo_codec",
]


def seed_of(*parts) -> int:
    """Deterministic 63-bit seed from any tuple of ints/strings."""
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


@dataclass(frozen=True)
class Op:
    """One step of a workload script.

    kind:
      'new'    -- create empty root branch ``branches[0]``
      'append' -- append ``n_new`` tokens to every branch in ``branches`` (one call)
      'fork'   -- fork each parent in ``branches``; parent i gets the children
                  ``children[i]`` (a tuple of new logical ids)
      'free'   -- release every branch in ``branches`` (one call)
      'truncate' -- roll branch i of ``branches`` back to ``new_lens[i]`` tokens (one call)
    """
    kind: str
    branches: Tuple[int, ...]
    n_new: int = 0
    children: Tuple[Tuple[int, ...], ...] = ()
    new_lens: Tuple[int, ...] = ()


@dataclass
class Workload:
    name: str
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    ops: List[Op]
    query: Tuple[int, ...]          # logical ids queried, in output order
    q_len: int = 1
    seed: int = 0                   # value seed (Q/K/V)
    meta: Dict[str, object] = field(default_factory=dict)

    # ---------------------------------------------------------------- values
    def kv(self, op_index: int, device="cpu", layer: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
        """K, V for append op ``op_index``: ``[n_branches][n_new][n_kv][d]``.

        Each branch's slice is drawn from its own generator, so any slice can
        be regenerated alone (:meth:`kv_one`).  ``layer`` selects the model
        layer (each layer draws its own values)."""
        op = self.ops[op_index]
        assert op.kind == "append"
        nb = len(op.branches)
        K = torch.empty((nb, op.n_new, self.n_kv_heads, self.head_dim), dtype=self.dtype, device=device)
        V = torch.empty_like(K)
        for i in range(nb):
            k, v = self.kv_one(op_index, i, device, layer)
            K[i].copy_(k)
            V[i].copy_(v)
        return K, V

    def kv_layers(self, op_index: int, n_layers: int, device="cpu") -> Tuple[torch.Tensor, torch.Tensor]:
        """K, V of every layer: ``[n_layers][n_branches][n_new][n_kv][d]``."""
        kv = [self.kv(op_index, device, l) for l in range(n_layers)]
        return torch.stack([k for k, _ in kv]), torch.stack([v for _, v in kv])

    def kv_one(self, op_index: int, pos: int, device="cpu", layer: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
        """K, V slice ``[n_new][n_kv][d]`` of the ``pos``-th branch of an append op."""
        op = self.ops[op_index]
        g = torch.Generator(device=device)
        # layer 0 keeps the single-layer seed, so one-layer runs are unchanged
        g.manual_seed(seed_of(self.seed, "kv", op_index, pos) if layer == 0 else
                      seed_of(self.seed, "kv", op_index, pos, "layer", layer))
        x = torch.randn((2, op.n_new, self.n_kv_heads, self.head_dim), generator=g,
                        device=device, dtype=torch.float32)
        x = x.to(self.dtype)
        return x[0], x[1]

    def q(self, device="cpu") -> torch.Tensor:
        """Queries ``[n_query][q_len][n_q_heads][d]``."""
        out = torch.empty((len(self.query), self.q_len, self.n_q_heads, self.head_dim),
                          dtype=self.dtype, device=device)
        for i in range(len(self.query)):
            out[i].copy_(self.q_one(i, device))
        return out

    def q_one(self, pos: int, device="cpu") -> torch.Tensor:
        g = torch.Generator(device=device)
        g.manual_seed(seed_of(self.seed, "q", pos))
        x = torch.randn((self.q_len, self.n_q_heads, self.head_dim), generator=g,
                        device=device, dtype=torch.float32)
        return x.to(self.dtype)

    # ------------------------------------------------------------ accounting
    def lengths(self) -> Dict[int, int]:
        """Token count of every live logical branch at the end of the script."""
        ln: Dict[int, int] = {}
        for op in self.ops:
            if op.kind == "new":
                ln[op.branches[0]] = 0
            elif op.kind == "append":
                for b in op.branches:
                    ln[b] += op.n_new
            elif op.kind == "fork":
                for p, ch in zip(op.branches, op.children):
                    for c in ch:
                        ln[c] = ln[p]
            elif op.kind == "free":
                for b in op.branches:
                    del ln[b]
            elif op.kind == "truncate":
                for b, n in zip(op.branches, op.new_lens):
                    ln[b] = n
        return ln

    def n_branch_ids(self) -> int:
        n = 0
        for op in self.ops:
            if op.kind == "new":
                n = max(n, op.branches[0] + 1)
            elif op.kind == "fork":
                for ch in op.children:
                    n = max(n, max(ch) + 1)
        return n

    def blocks_upper_bound(self) -> int:
        """Blocks a pool needs for the script: every block boundary crossed by
        an append plus one possible copy of a partial tail per appended branch."""
        ln: Dict[int, int] = {}
        total = 0
        bs = self.block_size
        for op in self.ops:
            if op.kind == "new":
                ln[op.branches[0]] = 0
            elif op.kind == "append":
                for b in op.branches:
                    L = ln[b]
                    total += -(-(L + op.n_new) // bs) - (-(-L // bs)) + (1 if L % bs else 0)
                    ln[b] = L + op.n_new
            elif op.kind == "fork":
                for p, ch in zip(op.branches, op.children):
                    for c in ch:
                        ln[c] = ln[p]
            elif op.kind == "truncate":
                for b, n in zip(op.branches, op.new_lens):
                    ln[b] = n
        return total

    def unique_kv_tokens(self) -> int:
        """Distinct stored token positions visible to the queried branches.

        A token is identified by the branch that appended it and its position;
        forks share everything before the fork point (Dendrite article, section
        "技术深度解析": the shared prefix is stored once)."""
        # nodes are (branch id, version); a truncate starts a new version of
        # the branch cut from the old one at the new length
        parent: Dict[Tuple[int, int], Tuple[Tuple[int, int], int]] = {}
        ln: Dict[Tuple[int, int], int] = {}
        cur: Dict[int, Tuple[int, int]] = {}
        for op in self.ops:
            if op.kind == "new":
                cur[op.branches[0]] = (op.branches[0], 0)
                ln[cur[op.branches[0]]] = 0
            elif op.kind == "append":
                for b in op.branches:
                    ln[cur[b]] += op.n_new
            elif op.kind == "fork":
                for p, ch in zip(op.branches, op.children):
                    for c in ch:
                        cur[c] = (c, 0)
                        parent[cur[c]] = (cur[p], ln[cur[p]])
                        ln[cur[c]] = ln[cur[p]]
            elif op.kind == "truncate":
                for b, n in zip(op.branches, op.new_lens):
                    old = cur[b]
                    cur[b] = (b, old[1] + 1)
                    parent[cur[b]] = (old, n)
                    ln[cur[b]] = n
        # Owner intervals: token position pos of branch b belongs to b when it
        # is at or beyond b's fork point, else to the parent (recursively).
        seen = set()
        for b in self.query:
            node = cur[b]
            cap = ln[node]
            while True:
                start = parent[node][1] if node in parent else 0
                if start < cap:
                    seen.update((node, pos) for pos in range(start, cap))
                if node not in parent:
                    break
                cap = min(cap, start)
                node = parent[node][0]
        return len(seen)

    def unique_kv_bytes(self) -> int:
        elt = torch.tensor([], dtype=self.dtype).element_size()
        return self.unique_kv_tokens() * 2 * self.n_kv_heads * self.head_dim * elt


# ====================================================================== scripts

def _roots(ops: List[Op], n: int, start: int = 0) -> List[int]:
    ids = list(range(start, start + n))
    for i in ids:
        ops.append(Op("new", (i,)))
    return ids


def tiny_cow(variant: str = "a", seed: int = 0) -> Workload:
    """The tiny copy-on-write fork check: fp32, 2 KV heads, 4 Q heads, head_dim
    64, block_size 16, a 64-token shared prefix forked into 2 branches that
    append 16 tokens each, one decode query per branch.

    Variant 'a' is the setting as stated (the 64-token prefix is block aligned,
    so no copy happens).  Variant 'b' appends 8 more tokens to the root before
    the fork, so the shared tail block is half full and both children must copy
    it (the root stays live).  Variant 'c' is 'b' with the root freed before the
    appends, so the first child copies and the second writes in place."""
    ops: List[Op] = [Op("new", (0,)), Op("append", (0,), 64)]
    if variant in ("b", "c"):
        ops.append(Op("append", (0,), 8))
    ops.append(Op("fork", (0,), children=((1, 2),)))
    if variant == "c":
        ops.append(Op("free", (0,)))
    ops.append(Op("append", (1, 2), 16))
    return Workload(f"tiny_{variant}", 2, 4, 64, 16, torch.float32, ops, (1, 2), 1, seed,
                    meta={"variant": variant})


def beam(requests=8, prefix=4096, width=4, divergent=256, n_kv=8, n_q=32, d=128,
         bs=16, dtype=torch.bfloat16, seed=0) -> Workload:
    """Beam-like 4-way fork: ``requests`` independent prompts of ``prefix``
    tokens, each forked ``width`` ways, each branch appending ``divergent``
    tokens, one decode query per branch."""
    ops: List[Op] = []
    roots = _roots(ops, requests)
    ops.append(Op("append", tuple(roots), prefix))
    nxt = requests
    children = []
    for _ in roots:
        children.append(tuple(range(nxt, nxt + width)))
        nxt += width
    ops.append(Op("fork", tuple(roots), children=tuple(children)))
    leaves = tuple(c for ch in children for c in ch)
    if divergent:
        ops.append(Op("append", leaves, divergent))
    return Workload(f"beam_r{requests}_p{prefix}_w{width}_div{divergent}", n_kv, n_q, d, bs,
                    dtype, ops, leaves, 1, seed,
                    meta=dict(requests=requests, prefix=prefix, width=width, divergent=divergent))


def mcts(root=2048, iters=500, width=4, per_node=32, max_depth=12, n_kv=8, n_q=32, d=128,
         bs=16, dtype=torch.bfloat16, seed=0, tree_seed=1) -> Workload:
    """MCTS-style tree (dendrite demo.tape, section "MCTS demo"): a ``root``
    token prompt; each iteration picks a uniformly random live leaf whose depth
    is below ``max_depth`` and forks it ``width`` ways, each child appending
    ``per_node`` tokens.  One decode query per live leaf at the end.  The
    selection policy is a uniform random stand-in (no model is run)."""
    rng = random.Random(seed_of(tree_seed, "mcts"))
    ops: List[Op] = [Op("new", (0,)), Op("append", (0,), root)]
    depth = {0: 0}
    leaves = [0]
    nxt = 1
    for _ in range(iters):
        cand = [b for b in leaves if depth[b] < max_depth]
        if not cand:
            break
        p = cand[rng.randrange(len(cand))]
        ch = tuple(range(nxt, nxt + width))
        nxt += width
        ops.append(Op("fork", (p,), children=(ch,)))
        ops.append(Op("append", ch, per_node))
        leaves.remove(p)
        for c in ch:
            depth[c] = depth[p] + 1
            leaves.append(c)
    q = tuple(sorted(leaves))
    return Workload(f"mcts_root{root}_it{iters}", n_kv, n_q, d, bs, dtype, ops, q, 1, seed,
                    meta=dict(root=root, iters=iters, width=width, per_node=per_node,
                              max_depth=max_depth, tree_seed=tree_seed,
                              mean_leaf_depth=sum(depth[b] for b in q) / len(q)))


def spec_verify(requests=32, prefix=8192, paths=3, draft=8, n_kv=8, n_q=32, d=128, bs=16,
                dtype=torch.bfloat16, seed=0) -> Workload:
    """Speculative-verification tree: ``paths`` draft paths of ``draft`` tokens
    forked at the end of each request's prefix; every draft token is a query
    (q_len = draft) that sees the prefix and its own path up to itself."""
    ops: List[Op] = []
    roots = _roots(ops, requests)
    ops.append(Op("append", tuple(roots), prefix))
    nxt = requests
    children = []
    for _ in roots:
        children.append(tuple(range(nxt, nxt + paths)))
        nxt += paths
    ops.append(Op("fork", tuple(roots), children=tuple(children)))
    leaves = tuple(c for ch in children for c in ch)
    ops.append(Op("append", leaves, draft))
    return Workload(f"specverify_r{requests}_p{prefix}_paths{paths}_q{draft}", n_kv, n_q, d, bs,
                    dtype, ops, leaves, draft, seed,
                    meta=dict(requests=requests, prefix=prefix, paths=paths, draft=draft))


def fork_stress_attention(requests=16, prefix=32768, width=64, divergent=1024, **kw) -> Workload:
    """Large fork stress: same shape as :func:`beam` at a 32K prefix and 64-way fork."""
    w = beam(requests=requests, prefix=prefix, width=width, divergent=divergent, **kw)
    w.name = f"stress_r{requests}_p{prefix}_w{width}_div{divergent}"
    return w


def fork_chain_script(depth_blocks: int, block_size: int = 16) -> int:
    """Length (tokens) of a chain of ``depth_blocks`` blocks whose tail block is
    half full: the fork-latency chains of the pages' fork_vs_depth benchmark
    (dendrite demo.tape, section "Fork benchmark results"), with depth read as
    the number of blocks."""
    return depth_blocks * block_size - block_size // 2


def random_script(rng_seed: int, n_ops: int = 40, max_live: int = 8, max_append: int = 40,
                  n_kv=2, n_q=4, d=16, bs=4, dtype=torch.float32, q_len=1, seed=0,
                  truncates: bool = False) -> Workload:
    """A random op sequence (fork / append / free) over a small pool, for
    property tests.  Appends pick several distinct live branches at once."""
    rng = random.Random(seed_of(rng_seed, "script"))
    ops: List[Op] = [Op("new", (0,))]
    live = [0]
    ln = {0: 0}
    nxt = 1
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.45 or not live:
            if not live:
                ops.append(Op("new", (nxt,)))
                live.append(nxt)
                ln[nxt] = 0
                nxt += 1
                continue
            k = rng.randint(1, min(3, len(live)))
            tgt = tuple(rng.sample(live, k))
            n = rng.randint(0, max_append)
            ops.append(Op("append", tgt, n))
            for b in tgt:
                ln[b] += n
        elif r < 0.75 and len(live) < max_live:
            p = rng.choice(live)
            nc = rng.randint(1, max(1, min(3, max_live - len(live))))
            ch = tuple(range(nxt, nxt + nc))
            nxt += nc
            ops.append(Op("fork", (p,), children=(ch,)))
            for c in ch:
                live.append(c)
                ln[c] = ln[p]
        elif r < 0.85 and len(live) > 1:
            b = rng.choice(live)
            ops.append(Op("free", (b,)))
            live.remove(b)
            del ln[b]
        elif r < 0.92 and truncates:
            k = rng.randint(1, min(2, len(live)))
            tgt = tuple(rng.sample(live, k))
            nl = tuple(rng.randint(0, ln[b]) for b in tgt)
            ops.append(Op("truncate", tgt, new_lens=nl))
            for b, n in zip(tgt, nl):
                ln[b] = n
        else:
            ops.append(Op("new", (nxt,)))
            live.append(nxt)
            ln[nxt] = 0
            nxt += 1
    # make every live branch long enough to be queried
    short = tuple(b for b in live if ln[b] < q_len)
    if short:
        ops.append(Op("append", short, q_len))
        for b in short:
            ln[b] += q_len
    return Workload(f"random_{rng_seed}", n_kv, n_q, d, bs, dtype, ops, tuple(sorted(live)),
                    q_len, seed)


def turbo_codec(seed: int = 0, head_dim: int = 128, qjl_rows: int = 128):
    """The random draws of a compressed pool's codec, seeded: rotation signs
    (float32 [head_dim], each +1 or -1) and the QJL matrix (float32
    [qjl_rows][head_dim], i.i.d. N(0, 1))."""
    g = torch.Generator().manual_seed(seed_of(seed, "turbo"))
    signs = (torch.randint(0, 2, (head_dim,), generator=g) * 2 - 1).to(torch.float32)
    S = torch.randn((qjl_rows, head_dim), generator=g, dtype=torch.float32)
    return signs, S
