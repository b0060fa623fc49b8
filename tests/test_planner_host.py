"""The host sharing planner (pure C function, no GPU) against the definition
of sharing: after a fork at t the child keeps the parent's blocks below
floor(t / block_size) for good (Dendrite article, ainews.cool, section
技术深度解析: positions 0..t-1 stay shared, positions >= t go to new leaves)."""
import random

import pytest

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.dendrite import plan_segments


def tree_arrays(w):
    """parent / fork_len / len over logical ids of a workload script."""
    n = w.n_branch_ids()
    parent, fork_len, ln = [-1] * n, [0] * n, [0] * n
    for op in w.ops:
        if op.kind == "append":
            for b in op.branches:
                ln[b] += op.n_new
        elif op.kind == "fork":
            for p, ch in zip(op.branches, op.children):
                for c in ch:
                    parent[c], fork_len[c], ln[c] = p, ln[p], ln[p]
    return parent, fork_len, ln


def owner(parent, fork_len, b, i, bs):
    while parent[b] >= 0 and i < fork_len[b] // bs:
        b = parent[b]
    return b


def check_plan(w, queried):
    parent, fork_len, ln = tree_arrays(w)
    bs = w.block_size
    segs = plan_segments(parent, fork_len, ln, bs, queried)
    cover = {}
    for rep, start, count, members in segs:
        assert count > 0 and members
        assert queried[members[0]] == rep
        for i in range(start, start + count):
            owners = {owner(parent, fork_len, queried[m], i, bs) for m in members}
            assert len(owners) == 1          # one physical block for all members
            for m in members:
                assert (m, i) not in cover    # each (branch, block) read once
                cover[(m, i)] = True
    for qi, b in enumerate(queried):
        for i in range(-(-ln[b] // bs)):
            assert (qi, i) in cover
    # every branch pair that shares a block owner reads it through the same segment
    for rep, start, count, members in segs:
        for i in range(start, start + count):
            o = owner(parent, fork_len, queried[members[0]], i, bs)
            same = [qi for qi, b in enumerate(queried) if i < -(-ln[b] // bs) and owner(parent, fork_len, b, i, bs) == o]
            assert sorted(same) == sorted(members)
    return segs


def test_beam_plan_reads_each_prefix_once():
    w = W.beam(requests=3, prefix=100, width=4, divergent=20)
    segs = check_plan(w, list(w.query))
    shared = [s for s in segs if len(s[3]) > 1]
    assert len(shared) == 3 and all(s[1] == 0 and s[2] == 100 // 16 and len(s[3]) == 4 for s in shared)


def test_mcts_plan():
    w = W.mcts(root=64, iters=40, width=4, per_node=8, max_depth=5)
    segs = check_plan(w, list(w.query))
    assert len(segs) > 10


@pytest.mark.parametrize("seed", range(30))
def test_random_trees(seed):
    w = W.random_script(seed, n_ops=30, max_live=8, max_append=40, bs=4)
    parent, fork_len, ln = tree_arrays(w)
    live = sorted(w.lengths().keys())
    rng = random.Random(seed)
    q = rng.sample(live, rng.randint(1, len(live)))
    check_plan(w, q)


def test_rejects_cycles_and_duplicates():
    from copy_write_forked_gb300.dendrite import DendriteError
    with pytest.raises(DendriteError):
        plan_segments([1, 0], [0, 0], [4, 4], 4, [0])
    with pytest.raises(DendriteError):
        plan_segments([-1], [0], [4], 4, [0, 0])
