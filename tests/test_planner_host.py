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


# ---------------------------------------------------------------- packing
# A packed segment reads its shared range with all its members and its extra
# tiles each with a subset of them; the attention result depends on the same
# two facts as for folding: every (queried branch, logical block) pair is read
# exactly once, and each tile is one physical block for every member that
# reads it (one owner by the walk of the sharing definition).

def check_packed(w, queried, rows_per_member, tc_min_rows=0, fold_pct=0, pack_pct=0):
    from copy_write_forked_gb300.dendrite import plan_segments_packed
    parent, fork_len, ln = tree_arrays(w)
    bs = w.block_size
    segs = plan_segments_packed(parent, fork_len, ln, bs, queried, rows_per_member, tc_min_rows=tc_min_rows,
                                fold_pct=fold_pct, pack_pct=pack_pct)
    cover = {}
    for rep, start, count, members, extras in segs:
        assert count > 0 and members and members == sorted(members)
        assert queried[members[0]] == rep
        for i in range(start, start + count):
            assert len({owner(parent, fork_len, queried[m], i, bs) for m in members}) == 1
            for m in members:
                assert (m, i) not in cover
                cover[(m, i)] = True
        if extras:
            assert len(members) <= 32
            rows = len(members) * rows_per_member
            assert rows <= (256 if tc_min_rows >= 0 and rows > (tc_min_rows or 64) else 64)
        for xrep, blk, mask in extras:
            readers = [members[k] for k in range(len(members)) if mask >> k & 1]
            assert readers and mask < (1 << len(members))
            assert xrep in [queried[m] for m in readers]
            o = owner(parent, fork_len, xrep, blk, bs)
            for m in readers:
                assert blk < -(-ln[queried[m]] // bs)
                assert owner(parent, fork_len, queried[m], blk, bs) == o
                assert (m, blk) not in cover
                cover[(m, blk)] = True
    assert len(cover) == sum(-(-ln[b] // bs) for b in queried)
    return segs


@pytest.mark.parametrize("seed", range(30))
def test_random_trees_pack_everything(seed):
    # pack_pct far above 100 packs every segment whose followers allow it
    w = W.random_script(seed, n_ops=40, max_live=10, max_append=40, bs=4)
    live = sorted(w.lengths().keys())
    rng = random.Random(seed)
    q = rng.sample(live, rng.randint(1, len(live)))
    for rpm in (1, 4, 24):
        for fold in (-1, 0, 1_000_000):
            check_packed(w, q, rpm, fold_pct=fold, pack_pct=1_000_000)
        check_packed(w, q, rpm, tc_min_rows=-1, pack_pct=1_000_000)


@pytest.mark.parametrize("seed", range(10))
def test_random_trees_default_pack(seed):
    w = W.random_script(seed, n_ops=60, max_live=12, max_append=20, bs=4)
    live = sorted(w.lengths().keys())
    check_packed(w, live, 4)
    check_packed(w, live, 32, tc_min_rows=-1)


def test_pack_off_is_the_folded_plan():
    w = W.mcts(root=64, iters=40, width=4, per_node=8, max_depth=5)
    parent, fork_len, ln = tree_arrays(w)
    q = list(w.query)
    packed = check_packed(w, q, 4, pack_pct=-1)
    assert [s[:4] for s in packed] == plan_segments(parent, fork_len, ln, 16, q, rows_per_member=4)
    assert all(not s[4] for s in packed)


def test_spec_verify_paths_pack_into_their_prefix():
    # 3 draft paths of 8 tokens (q_len 8, 32 rows each) below an 8192-token
    # prefix: the paths' one block each joins the prefix's 96-row unit
    w = W.spec_verify(requests=4)
    segs = check_packed(w, list(w.query), 32)
    assert len(segs) == 4
    for rep, start, count, members, extras in segs:
        assert (start, count, len(members)) == (0, 512, 3)
        assert sorted(m for _, _, m in extras) == [1, 2, 4]


def test_beam_leaves_pack_into_their_prefix_only_when_forced():
    # 16-block leaves of 4 rows under a 256-block prefix: packing saves their
    # unit starts, but every extra tile also costs the producer a dependent
    # load, so by default the leaves keep their own units
    w = W.beam(requests=2, prefix=4096, width=4, divergent=256)
    segs = check_packed(w, list(w.query), 4, pack_pct=1_000_000)
    assert len(segs) == 2 and all(len(s[4]) == 4 * 16 for s in segs)
    assert all(not s[4] for s in check_packed(w, list(w.query), 4))


def test_chains_are_folded_not_packed():
    # a branch's own range followed by its own tail segment (the same single
    # member): folding joins them without masks
    w = W.fork_stress_attention(requests=1, width=4, prefix=512, divergent=64)
    q = list(w.query)
    parent, fork_len, ln = tree_arrays(w)
    # each queried leaf forks one child that takes over the query
    n = len(parent)
    kids = []
    for i, b in enumerate(q):
        parent.append(b)
        fork_len.append(ln[b] - 3)
        ln.append(ln[b] - 3 + 1)
        kids.append(n + i)
    from copy_write_forked_gb300.dendrite import plan_segments_packed
    segs = plan_segments_packed(parent, fork_len, ln, w.block_size, kids, 4, pack_pct=1_000_000)
    assert all(not s[4] for s in segs)


def test_long_private_tails_do_not_pack():
    # the stress leaves (1024 tokens, 4 rows each) would be multiplied with the
    # prefix's 256 rows
    w = W.fork_stress_attention(requests=1, width=64)
    segs = check_packed(w, list(w.query), 4)
    assert all(not s[4] for s in segs) and len(segs) == 65


def test_mcts_packs_leaf_families():
    w = W.mcts()
    segs = check_packed(w, list(w.query), 4)
    folded = plan_segments(*tree_arrays(w), 16, list(w.query), rows_per_member=4)
    assert len(segs) * 2 < len(folded)
