"""Replays a workload script (see :mod:`.workloads`) through the C-ABI library.

Only marshalling: every operation is one library call (fork, append, free),
and the library returns the handles that logical ids map to."""
from __future__ import annotations

from typing import Dict, Optional

import torch

from .dendrite import Pool


def run_script(pool: Pool, w, device="cuda", stop: Optional[int] = None, stream=None,
               split_layers: bool = False, layer_order=None, start: int = 0,
               handles: Optional[Dict[int, int]] = None) -> Dict[int, int]:
    """Replays ``w`` on ``pool`` (ops ``start`` .. ``stop``; ``handles`` maps
    the logical ids of earlier ops, and is updated in place).  On a pool of
    several layers every append carries all layers: in one call, or with
    ``split_layers`` as ``append_begin`` followed by one ``append_layer`` per
    layer (in ``layer_order``, default ascending)."""
    h: Dict[int, int] = handles if handles is not None else {}
    nl = getattr(pool, "n_layers", 1)
    for idx, op in enumerate(w.ops[:stop]):
        if idx < start:
            continue
        if op.kind == "new":
            h[op.branches[0]] = pool.new_branch()
        elif op.kind == "fork":
            got = pool.fork_batch([h[p] for p in op.branches], [len(c) for c in op.children], stream=stream)
            for ch, handles in zip(op.children, got):
                for logical, handle in zip(ch, handles):
                    h[logical] = handle
        elif op.kind == "append":
            if op.n_new == 0:
                continue
            br = [h[b] for b in op.branches]
            if split_layers:
                pool.append_begin(br, op.n_new, stream=stream)
                for l in (layer_order if layer_order is not None else range(nl)):
                    K, V = w.kv(idx, device, layer=l)
                    pool.append_layer(l, K, V, stream=stream)
            elif nl == 1:
                K, V = w.kv(idx, device)
                pool.append_kv(br, K, V, stream=stream)
            else:
                K, V = w.kv_layers(idx, nl, device)
                pool.append_kv(br, K, V, stream=stream)
        elif op.kind == "free":
            pool.free([h[b] for b in op.branches], stream=stream)
            for b in op.branches:
                del h[b]
        elif op.kind == "truncate":
            pool.truncate([h[b] for b in op.branches], op.new_lens, stream=stream)
    return h


def _max_len(w) -> int:
    """Longest any branch gets during the script (rollbacks make it exceed the final lengths)."""
    ln, top = {}, 0
    for op in w.ops:
        if op.kind == "new":
            ln[op.branches[0]] = 0
        elif op.kind == "append":
            for b in op.branches:
                ln[b] += op.n_new
                top = max(top, ln[b])
        elif op.kind == "fork":
            for p, ch in zip(op.branches, op.children):
                for c in ch:
                    ln[c] = ln[p]
        elif op.kind == "truncate":
            for b, n in zip(op.branches, op.new_lens):
                ln[b] = n
    return top


def pool_for(w, extra_blocks: int = 16, max_branches: Optional[int] = None, **kw) -> Pool:
    """A pool sized for workload ``w``."""
    nb = max(1, w.blocks_upper_bound() + extra_blocks)
    mb = max_branches or max(16, w.n_branch_ids() + 8)
    bpb = max(16, -(-_max_len(w) // w.block_size) + 4)
    return Pool(nb, w.block_size, w.n_kv_heads, w.head_dim, w.dtype, max_branches=mb,
                max_blocks_per_branch=bpb, **kw)
