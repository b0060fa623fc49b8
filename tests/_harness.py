"""Helpers shared by the GPU parity tests: run a workload through the C-ABI
library and build the oracle's view of the same seeded inputs."""
from __future__ import annotations

from typing import Dict, Iterable, List, Set

import numpy as np
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.runner import pool_for, run_script
from oracle import KVTree
from oracle.block_pool import bits_of


def ancestors(w, ids: Iterable[int]) -> Set[int]:
    par = {}
    for op in w.ops:
        if op.kind == "fork":
            for p, ch in zip(op.branches, op.children):
                for c in ch:
                    par[c] = p
    out = set()
    for b in ids:
        while b is not None and b not in out:
            out.add(b)
            b = par.get(b)
    return out


def oracle_tree(w, ids: Iterable[int], device="cpu", layer: int = 0) -> KVTree:
    """O1 tree holding only the ancestor chains of ``ids``; each append slice
    is regenerated from its own seed on ``device`` (the values the GPU got),
    for model layer ``layer``."""
    keep = ancestors(w, ids)
    tree = KVTree(w.n_kv_heads, w.head_dim)
    for idx, op in enumerate(w.ops):
        if op.kind == "new" and op.branches[0] in keep:
            tree.new_root(op.branches[0])
        elif op.kind == "fork":
            for p, ch in zip(op.branches, op.children):
                if p in keep:
                    tree.fork(p, [c for c in ch if c in keep])
        elif op.kind == "append" and op.n_new:
            for pos, b in enumerate(op.branches):
                if b in keep:
                    k, v = w.kv_one(idx, pos, device, layer)
                    tree.append(b, k.cpu(), v.cpu())
        elif op.kind == "truncate":
            for b, n in zip(op.branches, op.new_lens):
                if b in keep:
                    tree.truncate(b, n)
    return tree


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) around |x|."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 8)


def check_attention(w, out: torch.Tensor, sample: List[int], tol: float, device="cuda",
                    strict: bool = False, layer: int = 0) -> float:
    """Max |GPU - oracle| over the sampled query positions (indices into w.query).

    ``tol`` bounds the arithmetic.  A bf16 output is also rounded to bf16 when
    stored, which alone can move it by half a bf16 ulp (up to 2^-8 |out|, so
    more than 5e-3 once |out| >= 1.28, as happens when a query sees one or two
    keys); unless ``strict``, that half ulp of the exact result is added to
    the bound element by element."""
    ids = [w.query[i] for i in sample]
    tree = oracle_tree(w, ids, device, layer)
    worst = 0.0
    for i in sample:
        q = w.q_one(i, device).cpu()
        ref = tree.attend(w.query[i], q)
        got = out[i].double().cpu().numpy()
        assert np.isfinite(got).all()
        err = np.abs(got - ref)
        bound = tol if (strict or out.dtype != torch.bfloat16) else tol + half_ulp_bf16(ref)
        worst = max(worst, float(err.max()))
        assert (err <= bound).all(), (w.name, i, float(err.max()), float((err - bound).max()))
    return worst


def pool_state_matches(pool, h: Dict[int, int], ref, check_bytes=True, layers=(0,)) -> None:
    """Bit-exact comparison of the device pool against the O2 model (the
    payload of every layer in ``layers``)."""
    for b, tab in ref.table.items():
        assert pool.read_table(h[b]) == tab, ("table", b)
    assert pool.read_refcounts() == ref.refcount.tolist()
    assert pool.read_free_stack() == ref.free_stack()
    if not check_bytes:
        return
    valid = {}
    for b, tab in ref.table.items():
        for pos in range(ref.len[b]):
            valid.setdefault(tab[pos // ref.bs], set()).add(pos % ref.bs)
    for layer in layers:
        for blk, slots in valid.items():
            k, v = pool.read_block(blk, layer=layer)
            kb, vb = bits_of(k), bits_of(v)
            sl = sorted(slots)
            assert np.array_equal(kb[:, sl], ref.KL[layer][blk][:, sl]), ("K bytes", layer, blk)
            assert np.array_equal(vb[:, sl], ref.VL[layer][blk][:, sl]), ("V bytes", layer, blk)
