"""Plain, slow fp64 CPU oracle for the copy-on-write tree KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) imports, links or executes this package; only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may.  It shares
no code with the CUDA path: the only common module is the seeded input
generator ``copy_write_forked_gb300.workloads``, which holds none of the
method's arithmetic.

Two models, both written from the pages' statement of the method:

* :mod:`oracle.kv_tree` (O1) -- the logical tree of the Dendrite article
  (ainews.cool, "Dendrite: O(1) KV cache forking", section "技术深度解析"):
  nodes hold token positions, a fork at position t creates empty leaves with a
  pointer back to the shared prefix, and attention gathers K/V from the shared
  ancestor path plus the branch's own leaf path.  Attention is
  softmax(q K^T / sqrt(d)) V in fp64 on the materialised sequence, and the
  log-sum-exp merge of partial (max, sum, acc) triples.
* :mod:`oracle.block_pool` (O2) -- a sequential model of the copy-on-write
  block table (dendrite demo.tape, section "The problem": "copy-on-write block
  table"): refcounted fixed-size blocks, a free stack, per-branch tables, the
  fork (table copy + refcount increment), the append that copies a shared
  partial tail block only when its refcount is above 1, and free.

* :mod:`oracle.turbo_quant` (O3) -- compressed KV rows (dendrite demo.tape,
  section "TurboQuant": "TurboQuant KV compression (PolarQuant + QJL)"):
  the pages give only the names, three test names and a ratio, so the steps
  follow the published methods they name (random Walsh-Hadamard rotation,
  the recursive polar transform with quantized angles, a one-bit QJL sketch
  of the key residual) and attention over the compressed rows.

Parity status: all three models are pinned (see ``tests/test_oracle_*.py``) by
brute force on tiny inputs, closed forms, invariants and hand-derived worked
states; no page prints a numeric attention output, so there is no printed
value to pin against.
"""
from .kv_tree import KVTree, lse_merge, partial_attention, run_script_tree  # noqa: F401
from .block_pool import BlockPool, PoolExhausted, run_script_pool  # noqa: F401
