"""Planning in fork-heavy loops, through the C-ABI library against the fp64
oracle at every step: the MCTS demo's loop (dendrite demo.tape, section "MCTS
demo": pick a leaf, fork it four ways, extend each child, then decode every
live leaf), where every iteration changes the queried set and so needs a new
plan, and decode loops whose appends cross into new blocks."""
import random

import numpy as np
import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.runner import pool_for
from oracle import KVTree

from _harness import half_ulp_bf16

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def _check(tree, leaf_ids, Q, out, sample):
    for i in sample:
        ref = tree.attend(leaf_ids[i], Q[i].cpu())
        got = out[i].double().cpu().numpy()
        err = np.abs(got - ref)
        assert np.isfinite(got).all()
        assert (err <= TOL + half_ulp_bf16(ref)).all(), (i, float(err.max()))


@pytest.mark.parametrize("fold,dev", [(0, 0), (-1, 0), (0, 1)])
def test_mcts_loop_matches_oracle_every_iteration(fold, dev):
    """60 iterations of fork 4 / append 32 / attend over every live leaf; each
    iteration's outputs are compared with the oracle's for the 4 new children
    and 4 other live leaves.  dev 1: every plan's units and CTA split are
    expanded on the device."""
    w = W.mcts(root=512, iters=60)
    pool = pool_for(w, fold_segments=fold, device_planning=dev)
    tree = KVTree(w.n_kv_heads, w.head_dim)
    gen = torch.Generator(device="cuda").manual_seed(5)
    h, live = {}, []
    rng = random.Random(3)
    iters = 0
    ops = w.ops
    i = 0
    while i < len(ops):
        op = ops[i]
        if op.kind == "new":
            h[op.branches[0]] = pool.new_branch()
            tree.new_root(op.branches[0])
            live.append(op.branches[0])
        elif op.kind == "append":
            K, V = w.kv(i, "cuda")
            pool.append_kv([h[b] for b in op.branches], K, V)
            for j, b in enumerate(op.branches):
                tree.append(b, K[j].cpu(), V[j].cpu())
        else:
            kids = pool.fork_batch([h[p] for p in op.branches], [len(c) for c in op.children])
            for p, ch, hs in zip(op.branches, op.children, kids):
                h.update(zip(ch, hs))
                tree.fork(p, list(ch))
                live.remove(p)
                live.extend(ch)
            nxt = ops[i + 1]
            K, V = w.kv(i + 1, "cuda")
            pool.append_kv([h[b] for b in nxt.branches], K, V)
            for j, b in enumerate(nxt.branches):
                tree.append(b, K[j].cpu(), V[j].cpu())
            q = sorted(live)
            Q = torch.randn((len(q), 1, w.n_q_heads, w.head_dim), generator=gen, device="cuda").bfloat16()
            out = pool.tree_attn_decode(Q, [h[b] for b in q])
            pool.sync()
            new = [q.index(c) for c in nxt.branches]
            others = rng.sample(range(len(q)), min(4, len(q)))
            _check(tree, q, Q, out, sorted(set(new + others)))
            iters += 1
            i += 1
        i += 1
    assert iters == 60
    pool.close()


def _extend(w, ops, query=None):
    return W.Workload(w.name + "_ext", w.n_kv_heads, w.n_q_heads, w.head_dim, w.block_size, w.dtype,
                      list(w.ops) + list(ops), tuple(query if query is not None else w.query), w.q_len, w.seed)


@pytest.mark.parametrize("step_tokens,dev,pack", [(1, 0, -1), (7, 0, -1), (23, 0, -1), (7, 1, -1), (7, 0, 0),
                                                   (23, 1, 0)])
def test_block_crossing_appends_lengthen_cached_segments(step_tokens, dev, pack):
    """Decode steps of 1, 7 or 23 tokens per branch: a step whose appends take
    branches into new blocks reuses the cached segments (stats.refreshed 2),
    with the same segments, tiles and partial rows as a plan built anew, and
    every step matches the oracle.  With the leaves packed into their prefix
    (pack 0) a branch's last blocks are extra tiles of the prefix's segment,
    read by it alone: the step adds extra tiles after them instead, and the
    plan keeps its packing even where a fresh build would no longer pack."""
    from _harness import check_attention
    from copy_write_forked_gb300.runner import run_script
    base = W.beam(requests=2, prefix=90, width=3, divergent=13)
    # enough steps to cross at least one block boundary (the leaves start at 103 tokens)
    steps = [W.Op("append", tuple(base.query), step_tokens) for _ in range(max(6, 24 // step_tokens))]
    w_full = _extend(base, steps)
    pool = pool_for(w_full, device_planning=dev, pack_segments=pack)
    h = run_script(pool, base)
    br = [h[b] for b in base.query]
    Q = base.q("cuda")
    pool.tree_attn_decode(Q, br)
    seen = set()
    for k in range(len(steps)):
        idx = len(base.ops) + k
        K, V = w_full.kv(idx, "cuda")
        pool.append_kv(br, K, V)
        out = pool.tree_attn_decode(Q, br)
        pool.sync()
        st = pool.last_plan_stats()
        seen.add(st["refreshed"])
        w_k = W.Workload(w_full.name, w_full.n_kv_heads, w_full.n_q_heads, w_full.head_dim, w_full.block_size,
                         w_full.dtype, w_full.ops[:idx + 1], w_full.query, w_full.q_len, w_full.seed)
        check_attention(w_k, out, list(range(len(base.query))), TOL)
        if st["refreshed"] == 2:
            # a plan built anew for the same tree (another query order misses the cache)
            perm = list(range(len(br)))[::-1]
            pool.tree_attn_decode(Q[perm].contiguous(), [br[i] for i in perm])
            fresh = pool.last_plan_stats()
            assert fresh["refreshed"] == 0
            # a packed plan grown in place keeps its packing while a fresh
            # build may no longer pack the longer leaves: then only the
            # distinct tiles must agree
            keys = ("n_segments", "n_units", "n_partials", "tiles", "unique_tiles") if pack < 0 else ("unique_tiles",)
            for key in keys:
                assert fresh[key] == st[key], key
            pool.tree_attn_decode(Q, br)          # the cached order again: a plain rebuild
            assert pool.last_plan_stats()["refreshed"] == 0
    assert 2 in seen
    pool.close()


def test_block_crossing_of_a_shared_last_segment_rebuilds():
    """A queried parent whose last block range is also read by a queried child
    (forked at its full, block-aligned length) is not lengthened in place: the
    step that takes the parent into a new block builds the plan anew."""
    from _harness import check_attention
    from copy_write_forked_gb300.runner import run_script
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 48), W.Op("fork", (0,), children=((1,),)),
           W.Op("append", (1,), 5)]
    base = W.Workload("shared_last", 2, 8, 128, 16, torch.bfloat16, ops, (0, 1))
    w_full = _extend(base, [W.Op("append", (0, 1), 1)])
    pool = pool_for(w_full)
    h = run_script(pool, base)
    br = [h[0], h[1]]
    Q = base.q("cuda")
    pool.tree_attn_decode(Q, br)
    K, V = w_full.kv(len(base.ops), "cuda")
    pool.append_kv(br, K, V)
    out = pool.tree_attn_decode(Q, br)
    pool.sync()
    assert pool.last_plan_stats()["refreshed"] == 0
    check_attention(w_full, out, [0, 1], TOL)
    pool.close()


STAT_KEYS = ("n_segments", "n_units", "n_ctas", "n_tc_ctas", "n_partials", "tiles", "unique_tiles")


def _device_cases():
    bf = dict(n_kv=8, n_q=32, d=128, bs=16, dtype=torch.bfloat16)
    return [
        ("mcts", lambda: W.mcts(root=512, iters=120)),
        ("beam", lambda: W.beam(requests=4, prefix=1024, width=4, divergent=64)),
        ("spec_verify", lambda: W.spec_verify(requests=4, prefix=2048)),
        ("fork_stress", lambda: W.fork_stress_attention(requests=2, prefix=4096, width=16, divergent=256)),
    ] + [(f"random_{k}", (lambda k=k: W.random_script(k, n_ops=60, max_live=24, max_append=300, **bf)))
         for k in range(6)]


@pytest.mark.parametrize("name,make", _device_cases(), ids=[c[0] for c in _device_cases()])
@pytest.mark.parametrize("fold", [0, -1])
def test_device_expansion_equals_host_expansion(name, make, fold):
    """The same call planned with the units and CTA split expanded on the
    device (device_planning 1) and on the host (-1): bit-identical outputs,
    the same CTA counts and partial rows, and oracle parity."""
    from _harness import check_attention
    from copy_write_forked_gb300.runner import run_script
    w = make()
    outs, stats = [], []
    for dev in (1, -1):
        pool = pool_for(w, fold_segments=fold, device_planning=dev)
        h = run_script(pool, w)
        br = [h[b] for b in w.query]
        Q = w.q("cuda")
        out = pool.tree_attn_decode(Q, br)
        pool.sync()
        outs.append(out.clone())
        stats.append(pool.last_plan_stats())
        # a second call on the unchanged tree reuses the plan (and its device copy)
        again = pool.tree_attn_decode(Q, br)
        pool.sync()
        assert torch.equal(again, out)
        pool.close()
    assert torch.equal(outs[0], outs[1]), name
    for key in STAT_KEYS:
        assert stats[0][key] == stats[1][key], (name, key, stats[0][key], stats[1][key])
    rng = random.Random(len(w.query))
    sample = sorted(rng.sample(range(len(w.query)), min(6, len(w.query))))
    check_attention(w, outs[0], sample, TOL)


def test_decode_loop_forking_every_leaf_keeps_the_tree_flat():
    """A decode loop that forks every leaf once per step, appends a token to
    each child and frees the old leaves (the bench's decode step): the host
    tree splices out the freed leaves' nodes, so the plan keeps the shape of
    the real forks (one segment per prefix and one per leaf, step after
    step) instead of growing a node per branch per step; the attention
    matches the oracle along the way."""
    from copy_write_forked_gb300.dendrite import Pool
    R, P, Wd, nkv, nq, d = 2, 200, 4, 8, 32, 128
    steps = 40
    pool = Pool(R * (P // 16 + 2) + R * Wd * (steps // 16 + 4) + 64, 16, nkv, d, torch.bfloat16,
                max_branches=R + 2 * R * Wd + 16, max_blocks_per_branch=(P + steps) // 16 + 8)
    tree = KVTree(nkv, d)
    gen = torch.Generator(device="cuda").manual_seed(11)

    def rows(n, t):
        return (torch.randn((n, t, nkv, d), generator=gen, device="cuda").bfloat16(),
                torch.randn((n, t, nkv, d), generator=gen, device="cuda").bfloat16())

    roots = [pool.new_branch() for _ in range(R)]
    ids = {h: h for h in roots}
    for h in roots:
        tree.new_root(h)
    K, V = rows(R, P)
    pool.append_kv(roots, K, V)
    for j, h in enumerate(roots):
        tree.append(h, K[j].cpu(), V[j].cpu())
    kids = pool.fork_batch(roots, [Wd] * R)
    leaves = []
    for h, ks in zip(roots, kids):
        tree.fork(h, ks)
        leaves.extend(ks)
    segs = []
    Q = torch.randn((len(leaves), 1, nq, d), generator=gen, device="cuda").bfloat16()
    for step in range(steps):
        kids = pool.fork_batch(leaves, [1] * len(leaves))
        br = [k[0] for k in kids]
        for lf, c in zip(leaves, br):
            tree.fork(lf, [c])
        K, V = rows(len(br), 1)
        pool.append_kv(br, K, V)
        for j, c in enumerate(br):
            tree.append(c, K[j].cpu(), V[j].cpu())
        out = pool.tree_attn_decode(Q, br)
        pool.sync()
        segs.append(pool.last_plan_stats()["n_segments"])
        if step in (0, 17, steps - 1):
            _check(tree, br, Q, out, range(len(br)))
        pool.free(leaves)
        for lf in leaves:
            tree.free(lf)
        leaves = br
    # one segment per prefix and one per leaf, or the leaves packed into
    # their prefix while they are short: never a chain that grows per step
    assert set(segs) <= {R, R + R * Wd}, segs
    pool.close()


@pytest.mark.parametrize("tc_sms", [-1, 0, 40, 100])
def test_sm_split_between_the_partial_kernels(tc_sms):
    """A tree with work for both partial kernels (a 64-way fork: 256 rows per
    KV head on the shared prefix, 4-row leaves) with the tcgen05 kernel given
    tc_sms SMs and the mma.sync kernel the others' CTA slots: the class CTA
    counts stay within the split, device and host expansion agree bit for
    bit, and the output matches the oracle."""
    from _harness import check_attention
    from copy_write_forked_gb300.runner import run_script
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = W.fork_stress_attention(requests=2, prefix=2048, width=64, divergent=120)
    outs, stats = [], []
    for dev in (1, -1):
        pool = pool_for(w, device_planning=dev, tc_sms=tc_sms)
        h = run_script(pool, w)
        out = pool.tree_attn_decode(w.q("cuda"), [h[b] for b in w.query])
        pool.sync()
        outs.append(out.clone())
        stats.append(pool.last_plan_stats())
        pool.close()
    assert torch.equal(outs[0], outs[1])
    for key in STAT_KEYS:
        assert stats[0][key] == stats[1][key], (key, stats[0][key], stats[1][key])
    st = stats[0]
    assert st["n_tc_units"] == 2 * 8 and st["n_ctas"] > 0
    if tc_sms > 0:
        assert st["n_tc_ctas"] <= tc_sms and st["n_ctas"] <= 2 * (sms - tc_sms)
    elif tc_sms < 0:
        assert st["n_tc_ctas"] > tc_sms and st["n_tc_ctas"] + st["n_ctas"] > sms
    check_attention(w, outs[0], list(range(0, len(w.query), 7)), TOL)


def test_packed_draft_paths_growing_past_the_extra_tile_limit():
    """Draft paths packed into their prefix's tcgen05 unit (96 rows) keep
    growing by a block per step: the cached plan adds their extra tiles while
    the unit stays within the tcgen05 kernel's limit of 64, then the plan is
    built anew (no longer packing the long paths); every checked step matches
    the oracle and the pool reports no error."""
    from _harness import check_attention
    from copy_write_forked_gb300.runner import run_script
    base = W.spec_verify(requests=1, prefix=600, paths=3, draft=8)
    steps = [W.Op("append", tuple(base.query), 16) for _ in range(24)]
    w_full = _extend(base, steps)
    pool = pool_for(w_full)
    h = run_script(pool, base)
    br = [h[b] for b in base.query]
    Q = base.q("cuda")
    out = pool.tree_attn_decode(Q, br)
    pool.sync()
    assert pool.last_plan_stats()["n_tc_units"] == 8
    seen = set()
    for k in range(len(steps)):
        idx = len(base.ops) + k
        K, V = w_full.kv(idx, "cuda")
        pool.append_kv(br, K, V)
        out = pool.tree_attn_decode(Q, br)
        pool.sync()
        st = pool.last_plan_stats()
        seen.add(st["refreshed"])
        if k in (0, 9, 19, 20, len(steps) - 1):
            w_k = W.Workload(w_full.name, w_full.n_kv_heads, w_full.n_q_heads, w_full.head_dim,
                             w_full.block_size, w_full.dtype, w_full.ops[:idx + 1], w_full.query, w_full.q_len,
                             w_full.seed)
            check_attention(w_k, out, list(range(len(base.query))), TOL)
    assert 2 in seen and 0 in seen, seen
    pool.close()
