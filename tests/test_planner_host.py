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


# ---------------------------------------------------------------- folding
# Folding makes segments no longer maximal, so the checks are what the
# attention result depends on: every (queried branch, logical block) pair is
# read exactly once, and every position of a segment is one physical block for
# all its members (one owner by the walk of the sharing definition).

def check_folded(w, queried, rows_per_member, tc_min_rows=0, fold_pct=0):
    parent, fork_len, ln = tree_arrays(w)
    bs = w.block_size
    segs = plan_segments(parent, fork_len, ln, bs, queried, rows_per_member=rows_per_member,
                         tc_min_rows=tc_min_rows, fold_pct=fold_pct)
    cover = {}
    for rep, start, count, members in segs:
        assert count > 0 and members and members == sorted(members)
        assert queried[members[0]] == rep
        for i in range(start, start + count):
            owners = {owner(parent, fork_len, queried[m], i, bs) for m in members}
            assert len(owners) == 1
            for m in members:
                assert (m, i) not in cover
                cover[(m, i)] = True
    n_pairs = sum(-(-ln[b] // bs) for b in queried)
    assert len(cover) == n_pairs
    return segs


def pair_count(segs):
    return sum(len(m) for _, _, _, m in segs)


@pytest.mark.parametrize("seed", range(30))
def test_random_trees_fold_everything(seed):
    # fold_pct far above 100 folds every segment that has a successor
    w = W.random_script(seed, n_ops=40, max_live=10, max_append=40, bs=4)
    live = sorted(w.lengths().keys())
    rng = random.Random(seed)
    q = rng.sample(live, rng.randint(1, len(live)))
    for rpm in (1, 4, 24):
        segs = check_folded(w, q, rpm, fold_pct=1_000_000)
        base = plan_segments(*tree_arrays(w), w.block_size, q)
        assert pair_count(segs) <= pair_count(base)


@pytest.mark.parametrize("seed", range(10))
def test_random_trees_default_fold(seed):
    w = W.random_script(seed, n_ops=60, max_live=12, max_append=20, bs=4)
    live = sorted(w.lengths().keys())
    check_folded(w, live, 4)
    check_folded(w, live, 32, tc_min_rows=-1)


def test_fold_off_is_the_sharing_plan():
    w = W.mcts(root=64, iters=40, width=4, per_node=8, max_depth=5)
    parent, fork_len, ln = tree_arrays(w)
    q = list(w.query)
    assert plan_segments(parent, fork_len, ln, 16, q, rows_per_member=4, fold_pct=-1) == \
        plan_segments(parent, fork_len, ln, 16, q)


def test_mcts_fold_drops_most_partial_rows():
    # 2048-token root, 500 forks into 4 children of 32 tokens: deep chains of
    # two-block segments, each of which would cost every row below it a partial
    w = W.mcts()
    base = plan_segments(*tree_arrays(w), 16, list(w.query))
    segs = check_folded(w, list(w.query), 4)
    assert pair_count(segs) * 3 < pair_count(base)


@pytest.mark.parametrize("make, rpm", [(lambda: W.beam(requests=2, prefix=4096, width=4, divergent=256), 4),
                                       (lambda: W.spec_verify(requests=2), 32),
                                       (lambda: W.fork_stress_attention(requests=1, width=64), 4)])
def test_long_shared_prefixes_are_not_folded(make, rpm):
    # re-reading a long prefix once per child costs far more than its partials
    w = make()
    parent, fork_len, ln = tree_arrays(w)
    q = list(w.query)
    assert plan_segments(parent, fork_len, ln, w.block_size, q, rows_per_member=rpm) == \
        plan_segments(parent, fork_len, ln, w.block_size, q)


def test_folded_rejects_bad_arguments():
    from copy_write_forked_gb300.dendrite import DendriteError
    with pytest.raises(DendriteError):
        plan_segments([-1], [0], [4], 4, [0], rows_per_member=1, tc_min_rows=-2)
    with pytest.raises(DendriteError):
        plan_segments([-1], [0], [4], 4, [0], rows_per_member=1, fold_pct=-2)
