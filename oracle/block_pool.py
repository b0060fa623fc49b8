"""O2: sequential model of the copy-on-write block pool.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources: dendrite demo.tape (section "The problem": Dendrite forks through a
"copy-on-write block table") and the Dendrite article (ainews.cool, section
"技术深度解析": the shared prefix is stored once; a fork at t shares positions
0..t-1 and gives each branch new, empty leaves for positions >= t; memory grows
only with the divergent tokens).

The model keeps K and V payload as raw bit patterns (uint16 for bf16, uint32
for fp32) so that copy-on-write copies and row writes can be compared bit for
bit.  Pool layout per block: ``[n_kv_heads][block_size][head_dim]``.

Readings where the pages are silent (each is the plainest one the rest
supports):

1. Allocation order: the free stack starts as S = [N-1, ..., 0] with top = N,
   and a pop returns S[top-1] (so block ids 0, 1, 2, ... are handed out first).
   Within one call branches are served in argument order; within a branch the
   copy of a shared partial tail comes first, then new blocks in position order.
2. Copy-on-write: before writing into a partially filled tail block, a branch
   copies it iff its refcount is above 1 *at that branch's turn* (branches of
   one call are handled as if one after the other).  Only the ``len % bs``
   valid slots are copied; the source loses one reference.
3. Free: a freed branch drops one reference on every block of its table; the
   blocks that reach zero in one call are pushed in descending id order, so a
   pool whose branches are all freed in one call returns to its initial state.
4. The parent of a fork stays live and keeps its references.
5. An append that would need more blocks than are free changes nothing and
   raises :class:`PoolExhausted` (all-or-nothing).
6. Layers (the pages describe one attention layer): a pool of n_layers keeps
   one K and one V array per layer, and one set of block ids, tables,
   refcounts and free stack for all of them, since every layer of a decoded
   token lives at the same position.  An append allocates once and writes
   (and copies on write) every layer.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np

__all__ = ["BlockPool", "PoolExhausted", "run_script_pool", "bits_of"]


class PoolExhausted(RuntimeError):
    pass


def bits_of(t) -> np.ndarray:
    """Raw bit pattern of a torch tensor (bf16 -> uint16, fp32 -> uint32)."""
    import torch
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    raise TypeError(f"unsupported dtype {t.dtype}")


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                 bits_dtype=np.uint16, n_layers: int = 1):
        self.N = num_blocks
        self.bs = block_size
        self.n_kv = n_kv_heads
        self.d = head_dim
        self.n_layers = n_layers
        # per layer [num_blocks][n_kv][block_size][head_dim]; K / V are layer 0
        self.KL = np.zeros((n_layers, num_blocks, n_kv_heads, block_size, head_dim), dtype=bits_dtype)
        self.VL = np.zeros_like(self.KL)
        self.K = self.KL[0]
        self.V = self.VL[0]
        self.refcount = np.zeros(num_blocks, dtype=np.int64)
        self.stack = list(range(num_blocks - 1, -1, -1))   # S[0..N-1]
        self.top = num_blocks
        self.table: Dict[int, List[int]] = {}
        self.len: Dict[int, int] = {}

    # -------------------------------------------------------------- stack
    def _pop(self) -> int:
        self.top -= 1
        return self.stack[self.top]

    def _push(self, blk: int) -> None:
        self.stack[self.top] = blk
        self.top += 1

    def free_stack(self) -> List[int]:
        """The live part of the free stack, bottom to top (S[0..top-1])."""
        return self.stack[:self.top]

    # ---------------------------------------------------------------- ops
    def new_branch(self, h: int) -> None:
        assert h not in self.table
        self.table[h] = []
        self.len[h] = 0

    def fork(self, parents: Sequence[int], children: Sequence[Sequence[int]]) -> None:
        """Each child gets a copy of its parent's block table and length; every
        block of the parent gains one reference per child.  No payload moves."""
        for p, chs in zip(parents, children):
            for c in chs:
                assert c not in self.table
                self.table[c] = list(self.table[p])
                self.len[c] = self.len[p]
            for blk in self.table[p]:
                self.refcount[blk] += len(chs)

    def _demand(self, branches: Sequence[int], n_new: int) -> int:
        """Blocks an append would pop, with the same sequential decisions."""
        rc = {}
        total = 0
        for b in branches:
            L = self.len[b]
            fill = L % self.bs
            if fill and n_new > 0:
                tail = self.table[b][L // self.bs]
                r = rc.get(tail, int(self.refcount[tail]))
                if r > 1:
                    total += 1
                    rc[tail] = r - 1
            total += -(-(L + n_new) // self.bs) - (-(-L // self.bs))
        return total

    def append(self, branches: Sequence[int], n_new: int, K_bits: np.ndarray,
               V_bits: np.ndarray) -> None:
        """Append ``n_new`` rows to every branch; ``K_bits``/``V_bits`` are
        ``[n_branches][n_new][n_kv][d]`` raw bit patterns, with a leading
        ``[n_layers]`` axis for a pool of several layers."""
        if len(set(branches)) != len(branches):
            raise ValueError("duplicate branch in one append")
        if n_new == 0:
            return
        K_bits = np.asarray(K_bits)
        V_bits = np.asarray(V_bits)
        if K_bits.ndim == 4:
            K_bits, V_bits = K_bits[None], V_bits[None]
        assert K_bits.shape[0] == self.n_layers
        if self._demand(branches, n_new) > self.top:
            raise PoolExhausted("not enough free blocks")
        bs = self.bs
        for i, b in enumerate(branches):
            L = self.len[b]
            tab = self.table[b]
            fill = L % bs
            if fill:
                tail = tab[L // bs]
                if self.refcount[tail] > 1:
                    new = self._pop()
                    self.KL[:, new, :, :fill] = self.KL[:, tail, :, :fill]
                    self.VL[:, new, :, :fill] = self.VL[:, tail, :, :fill]
                    self.refcount[tail] -= 1
                    self.refcount[new] = 1
                    tab[L // bs] = new
            for t in range(n_new):
                bi, slot = divmod(L + t, bs)
                if bi == len(tab):
                    new = self._pop()
                    self.refcount[new] = 1
                    tab.append(new)
                self.KL[:, tab[bi], :, slot] = K_bits[:, i, t]
                self.VL[:, tab[bi], :, slot] = V_bits[:, i, t]
            self.len[b] = L + n_new

    def free(self, branches: Sequence[int]) -> None:
        released = []
        for b in branches:
            for blk in self.table[b]:
                self.refcount[blk] -= 1
                assert self.refcount[blk] >= 0
                if self.refcount[blk] == 0:
                    released.append(blk)
            del self.table[b]
            del self.len[b]
        for blk in sorted(released, reverse=True):
            self._push(blk)

    def truncate(self, branches: Sequence[int], new_lens: Sequence[int]) -> None:
        """Roll each branch back to its first new_len tokens (speculative
        decoding's reject step: DSpark blog, section "第二层：预测 + 并行 + 验证
        + 回滚", Accept / Rollback).  Table entries past ceil(new_len / bs)
        drop one reference; the kept tail block, if partially valid now, is
        copied on the next append when still shared.  Released blocks of the
        call are pushed in descending id order, as for free."""
        if len(set(branches)) != len(branches):
            raise ValueError("duplicate branch in one truncate")
        for b, n in zip(branches, new_lens):
            if not 0 <= n <= self.len[b]:
                raise ValueError("new length out of range")
        released = []
        for b, n in zip(branches, new_lens):
            keep = -(-n // self.bs)
            for blk in self.table[b][keep:]:
                self.refcount[blk] -= 1
                if self.refcount[blk] == 0:
                    released.append(blk)
            del self.table[b][keep:]
            self.len[b] = n
        for blk in sorted(released, reverse=True):
            self._push(blk)

    # ---------------------------------------------------------- inspection
    def read_branch_bits(self, h: int, layer: int = 0):
        """K and V bits ``[len][n_kv][d]`` of branch ``h`` in ``layer``, read through its table."""
        L = self.len[h]
        K = np.empty((L, self.n_kv, self.d), dtype=self.K.dtype)
        V = np.empty_like(K)
        for pos in range(L):
            blk = self.table[h][pos // self.bs]
            K[pos] = self.KL[layer, blk, :, pos % self.bs]
            V[pos] = self.VL[layer, blk, :, pos % self.bs]
        return K, V

    def used_blocks(self) -> int:
        return self.N - self.top


def run_script_pool(w, num_blocks: int, kv_source=None, stop=None, n_layers: int = 1,
                    device="cpu") -> BlockPool:
    """Replay a workload script (logical ids as handles) on a fresh pool.
    ``stop``: replay only the first ``stop`` ops.  With ``n_layers`` > 1 an
    append carries every layer's rows (``w.kv(idx, device, layer=l)``;
    ``device`` picks the generator, so it must be where the GPU run drew its
    values)."""
    import torch
    bits = np.uint16 if w.dtype == torch.bfloat16 else np.uint32
    pool = BlockPool(num_blocks, w.block_size, w.n_kv_heads, w.head_dim, bits, n_layers)
    for idx, op in enumerate(w.ops[:stop]):
        if op.kind == "new":
            pool.new_branch(op.branches[0])
        elif op.kind == "fork":
            pool.fork(op.branches, op.children)
        elif op.kind == "append":
            if op.n_new == 0:
                continue
            if n_layers == 1:
                K, V = kv_source(idx) if kv_source else w.kv(idx)
                pool.append(op.branches, op.n_new, bits_of(K), bits_of(V))
            else:
                kv = [w.kv(idx, device, layer=l) for l in range(n_layers)]
                pool.append(op.branches, op.n_new, np.stack([bits_of(k) for k, _ in kv]),
                            np.stack([bits_of(v) for _, v in kv]))
        elif op.kind == "free":
            pool.free(op.branches)
        elif op.kind == "truncate":
            pool.truncate(op.branches, op.new_lens)
    return pool
