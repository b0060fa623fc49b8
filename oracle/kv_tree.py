"""O1: the logical copy-on-write KV tree and its decode attention, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: Dendrite article (ainews.cool, "Dendrite: O(1) KV cache forking",
section "技术深度解析").  The article states that

* the KV cache is organised as a tree whose nodes are token positions, and the
  prefix shared by every branch is stored once;
* forking at position t copies nothing for positions 0..t-1: each new branch
  gets a new, empty leaf for positions >= t plus a pointer back to the shared
  prefix;
* attention walks this tree and gathers keys and values from the shared
  ancestor path and from the branch's own leaf path.

This module is that model with no physical layout at all: a node keeps its
parent, the fork position t and the K/V rows it appended itself.  Attention
materialises the branch's full sequence (ancestor path cut at each fork
position, then the branch's own rows) and evaluates softmax(q K^T / sqrt(d)) V
with a max-subtracted softmax in fp64.

Readings where the pages are silent:

* scale 1/sqrt(head_dim);
* grouped-query attention: query head h reads KV head floor(h / G) with
  G = n_q_heads / n_kv_heads;
* a decode query sees every stored position of its branch; with q_len > 1 the
  queries are the last q_len positions and query j sees positions
  <= len - q_len + j (the draft tokens of one parallel verification, DSpark
  blog, section "第二层：预测 + 并行 + 验证 + 回滚");
* the parent stays live after a fork and may keep appending; its children see
  only its first t positions.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np

__all__ = ["KVTree", "partial_attention", "lse_merge", "attention_dense", "run_script_tree"]


def _f64(x) -> np.ndarray:
    """Exact conversion of a torch tensor / array (bf16, fp16, fp32, fp64) to fp64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


class _Node:
    __slots__ = ("parent", "fork_len", "k", "v")

    def __init__(self, parent, fork_len: int, n_kv: int, d: int):
        self.parent = parent          # _Node or None (a root)
        self.fork_len = fork_len      # t: positions 0..t-1 come from the parent
        self.k: List[np.ndarray] = []  # own rows, each [n_kv][d]
        self.v: List[np.ndarray] = []

    def length(self) -> int:
        return self.fork_len + len(self.k)


class KVTree:
    """Branch handles -> tree nodes.  Freed handles drop their name only; a
    node stays reachable from its descendants (their pointer back to the
    shared prefix)."""

    def __init__(self, n_kv_heads: int, head_dim: int):
        self.n_kv = n_kv_heads
        self.d = head_dim
        self.nodes: Dict[int, _Node] = {}

    # ------------------------------------------------------------------ ops
    def new_root(self, h: int) -> None:
        assert h not in self.nodes
        self.nodes[h] = _Node(None, 0, self.n_kv, self.d)

    def fork(self, parent: int, children: Sequence[int]) -> None:
        """Fork at t = current length of ``parent``: every child is an empty
        leaf that points back to the parent's first t positions."""
        p = self.nodes[parent]
        t = p.length()
        for c in children:
            assert c not in self.nodes
            self.nodes[c] = _Node(p, t, self.n_kv, self.d)

    def append(self, h: int, K, V) -> None:
        """Append rows ``K``/``V`` ``[n][n_kv][d]`` to branch ``h``'s own leaf."""
        K = _f64(K)
        V = _f64(V)
        node = self.nodes[h]
        for i in range(K.shape[0]):
            node.k.append(K[i].copy())
            node.v.append(V[i].copy())

    def free(self, h: int) -> None:
        del self.nodes[h]

    def truncate(self, h: int, n: int) -> None:
        """Roll branch ``h`` back to its first ``n`` positions (the reject step
        of one parallel verification, DSpark blog, section 第二层).  The branch
        continues as a new leaf cut from its old node at position n, so any
        child forked from the old node keeps seeing what it saw."""
        old = self.nodes[h]
        assert 0 <= n <= old.length()
        self.nodes[h] = _Node(old, n, self.n_kv, self.d)

    def length(self, h: int) -> int:
        return self.nodes[h].length()

    # ------------------------------------------------------------ attention
    def materialise(self, h: int) -> Tuple[np.ndarray, np.ndarray]:
        """Full K and V ``[len][n_kv][d]`` of branch ``h``: the ancestor path
        (each ancestor cut at the fork position) followed by its own rows."""
        return self._materialise(self.nodes[h])

    def _materialise(self, node: _Node) -> Tuple[np.ndarray, np.ndarray]:
        empty = np.zeros((0, self.n_kv, self.d))
        if node.parent is not None:
            pk, pv = self._materialise(node.parent)
            pk, pv = pk[:node.fork_len], pv[:node.fork_len]
        else:
            pk, pv = empty, empty
        ok = np.stack(node.k) if node.k else empty
        ov = np.stack(node.v) if node.v else empty
        return np.concatenate([pk, ok]), np.concatenate([pv, ov])

    def attend(self, h: int, Q) -> np.ndarray:
        """Decode attention of branch ``h`` for queries ``Q`` ``[q_len][n_q][d]``.

        Returns ``[q_len][n_q][d]`` fp64: softmax(q K^T / sqrt(d)) V over the
        positions each query sees."""
        K, V = self.materialise(h)
        return attention_dense(_f64(Q), K, V)


def attention_dense(Q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V for every query row, fp64.

    ``Q`` ``[q_len][n_q][d]`` are the last q_len positions of the sequence
    ``K``/``V`` ``[L][n_kv][d]``; query j sees positions 0..L-q_len+j."""
    q_len, n_q, d = Q.shape
    L, n_kv, _ = K.shape
    assert n_q % n_kv == 0 and L >= q_len
    G = n_q // n_kv
    out = np.empty((q_len, n_q, d))
    for j in range(q_len):
        vis = L - q_len + j + 1
        for hq in range(n_q):
            kv = hq // G
            s = K[:vis, kv, :] @ Q[j, hq] / math.sqrt(d)
            p = np.exp(s - s.max())
            out[j, hq] = (p @ V[:vis, kv, :]) / p.sum()
    return out


def partial_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """One split-KV partial for a single query row over a subset of keys.

    ``q`` ``[d]``, ``K``/``V`` ``[n][d]``.  Returns (m, l, acc): the max of the
    scaled scores, the sum of exp(score - m) and the exp-weighted sum of V rows
    (unnormalised).  An empty key subset gives (-inf, 0, 0)."""
    d = q.shape[0]
    if K.shape[0] == 0:
        return -math.inf, 0.0, np.zeros(V.shape[1] if V.ndim == 2 else d)
    s = K @ q / math.sqrt(d)
    m = float(s.max())
    p = np.exp(s - m)
    return m, float(p.sum()), p @ V


def lse_merge(parts) -> np.ndarray:
    """Log-sum-exp merge of partial triples (m_i, l_i, acc_i) of one row:
    M = max m_i, L = sum l_i e^(m_i - M), out = sum acc_i e^(m_i - M) / L."""
    ms = [m for m, _, _ in parts]
    M = max(ms)
    L = 0.0
    acc = None
    for m, l, a in parts:
        w = 0.0 if m == -math.inf else math.exp(m - M)
        L += l * w
        acc = a * w if acc is None else acc + a * w
    return acc / L


def run_script_tree(w, kv_source=None) -> KVTree:
    """Replay a :class:`copy_write_forked_gb300.workloads.Workload` script on a
    fresh :class:`KVTree` keyed by logical ids.  ``kv_source(op_index)``
    returns the (K, V) of an append op; it defaults to ``w.kv(op_index)``."""
    tree = KVTree(w.n_kv_heads, w.head_dim)
    for idx, op in enumerate(w.ops):
        if op.kind == "new":
            tree.new_root(op.branches[0])
        elif op.kind == "fork":
            for p, ch in zip(op.branches, op.children):
                tree.fork(p, ch)
        elif op.kind == "append":
            if op.n_new == 0:
                continue
            K, V = kv_source(idx) if kv_source else w.kv(idx)
            for i, b in enumerate(op.branches):
                tree.append(b, K[i], V[i])
        elif op.kind == "free":
            for b in op.branches:
                tree.free(b)
        elif op.kind == "truncate":
            for b, n in zip(op.branches, op.new_lens):
                tree.truncate(b, n)
    return tree
