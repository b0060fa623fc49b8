"""Device block pool against the sequential oracle O2, bit for bit: block
tables, refcounts, the free stack and the K/V bytes of every valid slot
(copy-on-write copies included).  Through the C-ABI library on cuda:0."""
import json
import os

import numpy as np
import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.dendrite import DendriteError, Pool
from copy_write_forked_gb300.runner import pool_for, run_script
from oracle.block_pool import BlockPool, PoolExhausted, bits_of, run_script_pool

from _harness import pool_state_matches

pytestmark = pytest.mark.gpu
GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_cow_states.json")))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def _gpu_kv(w):
    return lambda idx: w.kv(idx, "cuda")


@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_tiny_cow_golden_and_oracle(variant):
    w = W.tiny_cow(variant)
    g = GOLDEN["cases"][variant]
    pool = Pool(64, 16, 2, 64, torch.float32, max_branches=8, max_blocks_per_branch=16)
    h = run_script(pool, w)
    pool.sync()
    for b, tab in g["tables"].items():
        assert pool.read_table(h[int(b)]) == tab
        assert pool.branch_len(h[int(b)]) == g["lens"][b]
    rc = pool.read_refcounts()
    assert rc[:len(g["refcount_prefix"])] == g["refcount_prefix"] and sum(rc[len(g["refcount_prefix"]):]) == 0
    assert 64 - len(pool.read_free_stack()) == g["used_blocks"]
    for dst, src, fill in g["cow_copies"]:
        kd, vd = pool.read_block(dst)
        ks, vs = pool.read_block(src)
        assert torch.equal(kd[:, :fill], ks[:, :fill]) and torch.equal(vd[:, :fill], vs[:, :fill])
    ref = run_script_pool(w, 64, kv_source=_gpu_kv(w))
    pool_state_matches(pool, h, ref)
    pool.free(list(h.values()))
    pool.sync()
    assert sum(pool.read_refcounts()) == 0
    assert pool.read_free_stack() == list(range(63, -1, -1))
    pool.close()


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_random_scripts_match_oracle_after_every_op(seed, dtype):
    d = 128 if dtype == torch.bfloat16 else 32
    w = W.random_script(seed, n_ops=30, max_live=8, max_append=40, n_kv=2, n_q=4, d=d, bs=16, dtype=dtype)
    N = w.blocks_upper_bound() + 5
    pool = Pool(N, 16, 2, d, dtype, max_branches=64, max_blocks_per_branch=64)
    h = {}
    ref = BlockPool(N, 16, 2, d, np.uint16 if dtype == torch.bfloat16 else np.uint32)
    for idx, op in enumerate(w.ops):
        if op.kind == "new":
            h[op.branches[0]] = pool.new_branch()
            ref.new_branch(op.branches[0])
        elif op.kind == "fork":
            got = pool.fork_batch([h[p] for p in op.branches], [len(c) for c in op.children])
            for ch, hs in zip(op.children, got):
                h.update(zip(ch, hs))
            ref.fork(op.branches, op.children)
        elif op.kind == "append":
            if op.n_new:
                K, V = w.kv(idx, "cuda")
                pool.append_kv([h[b] for b in op.branches], K, V)
                ref.append(op.branches, op.n_new, bits_of(K), bits_of(V))
        elif op.kind == "free":
            pool.free([h[b] for b in op.branches])
            ref.free(op.branches)
            for b in op.branches:
                del h[b]
        pool.sync()
        pool_state_matches(pool, h, ref, check_bytes=(idx == len(w.ops) - 1 or idx % 7 == 0))
    pool.close()


def test_golden_truncate_case_on_gpu():
    g = GOLDEN["truncate_case"]
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 20), W.Op("fork", (0,), children=((1, 2),)),
           W.Op("append", (1,), 20), W.Op("append", (2,), 8), W.Op("truncate", (1, 2), new_lens=(22, 20)),
           W.Op("free", (0,)), W.Op("append", (1,), 3), W.Op("append", (2,), 1)]
    w = W.Workload("trunc", 2, 4, 64, 16, torch.float32, ops, (1, 2))
    pool = Pool(64, 16, 2, 64, torch.float32, max_branches=8, max_blocks_per_branch=16)
    h = run_script(pool, w)
    pool.sync()
    for b, tab in g["tables"].items():
        assert pool.read_table(h[int(b)]) == tab
    rc = pool.read_refcounts()
    assert rc[:len(g["refcount_prefix"])] == g["refcount_prefix"]
    assert pool.read_free_stack()[-2:] == g["free_stack_top"]
    ref = run_script_pool(w, 64, kv_source=_gpu_kv(w))
    pool_state_matches(pool, h, ref)
    pool.close()


@pytest.mark.parametrize("seed", range(10))
def test_random_scripts_with_rollbacks_match_oracle(seed):
    w = W.random_script(100 + seed, n_ops=30, max_live=8, max_append=40, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, truncates=True)
    pool = pool_for(w)
    h = run_script(pool, w)
    ref = run_script_pool(w, pool.num_blocks, kv_source=_gpu_kv(w))
    pool.sync()
    pool_state_matches(pool, h, ref)
    pool.close()


def test_three_holders_of_one_tail_follow_argument_order():
    # root of 40 tokens (tail half full) forked 3 ways, root freed: refcount 3 = holders,
    # so in argument order [c3, c1, c2] the first two copy and the last writes in place
    w = W.Workload("three", 2, 4, 128, 16, torch.bfloat16,
                   [W.Op("new", (0,)), W.Op("append", (0,), 40), W.Op("fork", (0,), children=((1, 2, 3),)),
                    W.Op("free", (0,)), W.Op("append", (3, 1, 2), 5)], (1, 2, 3))
    pool = pool_for(w)
    h = run_script(pool, w)
    ref = run_script_pool(w, pool.num_blocks, kv_source=_gpu_kv(w))
    pool.sync()
    pool_state_matches(pool, h, ref)
    assert ref.table[2][2] == 2 and ref.table[3][2] != 2 and ref.table[1][2] != 2
    pool.close()


@pytest.mark.parametrize("sizes,every", [((200, 150, 10), 3), ((800, 590, 10), 1)])
def test_large_fork_batches_match_oracle(sizes, every):
    """One fork call of 360 pairs (its arguments in kernel parameters) or of
    1,400 pairs (staged in device memory), then an append to every third
    child or to all 1,400: tables and refcounts match O2."""
    n = sum(sizes)
    bounds = [2, 2 + sizes[0], 2 + sizes[0] + sizes[1], 2 + n]
    w = W.Workload("wide", 1, 1, 128, 16, torch.bfloat16,
                   [W.Op("new", (0,)), W.Op("new", (1,)), W.Op("append", (0, 1), 77),
                    W.Op("fork", (0, 1, 0), children=tuple(tuple(range(bounds[k], bounds[k + 1])) for k in range(3))),
                    W.Op("append", tuple(range(2, 2 + n, every)), 9)], tuple(range(2, 2 + n)))
    pool = pool_for(w, max_branches=n + 40)
    h = run_script(pool, w)
    ref = run_script_pool(w, pool.num_blocks, kv_source=_gpu_kv(w))
    pool.sync()
    pool_state_matches(pool, h, ref, check_bytes=False)
    pool.close()


@pytest.mark.parametrize("n_leaves", [300, 600, 1400])
def test_batched_forks_and_frees_of_siblings_match_oracle(n_leaves):
    """The shape of a decode step over many leaves that share two prompts'
    prefixes: every step forks each leaf once (one call of n_leaves pairs),
    appends one token to every child (a copy of each leaf's partial tail) and
    frees the old leaves in one call; finally everything is freed in one
    call.  Calls of this size take the tiled free kernel, whose lanes drop
    the references of a block shared within a tile with one atomic; their
    arguments travel as kernel parameters (300, 600 leaves) or are staged in
    device memory (1,400).  Tables, refcounts, the free stack and every valid
    slot match O2 after each step, and the last free returns every block to
    the stack."""
    half = n_leaves // 2
    ops = [W.Op("new", (0,)), W.Op("new", (1,)), W.Op("append", (0, 1), 100),
           W.Op("fork", (0, 1), children=(tuple(range(2, 2 + half)), tuple(range(2 + half, 2 + n_leaves)))),
           W.Op("append", tuple(range(2, 2 + n_leaves)), 5)]
    leaves = list(range(2, 2 + n_leaves))
    nxt = 2 + n_leaves
    checkpoints = []
    for step in range(3):
        kids = tuple(range(nxt, nxt + len(leaves)))
        nxt += len(leaves)
        ops.append(W.Op("fork", tuple(leaves), children=tuple((c,) for c in kids)))
        ops.append(W.Op("append", kids, 1))
        ops.append(W.Op("free", tuple(leaves)))
        leaves = list(kids)
        checkpoints.append(len(ops))
    ops.append(W.Op("free", tuple([0, 1] + leaves)))
    checkpoints.append(len(ops))
    w = W.Workload("siblings", 2, 8, 128, 16, torch.bfloat16, ops, (0,))
    pool = pool_for(w, max_branches=nxt + 8)
    h = {}
    done = 0
    for stop in checkpoints:
        run_script(pool, w, stop=stop, start=done, handles=h)
        done = stop
        ref = run_script_pool(w, pool.num_blocks, kv_source=_gpu_kv(w), stop=stop)
        pool.sync()
        pool_state_matches(pool, h, ref)
    assert sorted(pool.read_free_stack()) == list(range(pool.num_blocks))
    assert sum(pool.read_refcounts()) == 0
    pool.close()


def test_fork_each_is_fork_batch_with_one_child_each():
    """Pool.fork_each(parents) forks one child per parent: the same tables,
    lengths and refcounts as fork_batch with every count 1, children in the
    parents' order; an empty call forks nothing."""
    states = []
    for use_each in (True, False):
        pool = Pool(64, 16, 2, 64, torch.float32, max_branches=16, max_blocks_per_branch=8)
        a, b = pool.new_branch(), pool.new_branch()
        K = torch.randn(2, 37, 2, 64, device="cuda")
        pool.append_kv([a, b], K, K)
        kids = pool.fork_each([b, a]) if use_each else [k[0] for k in pool.fork_batch([b, a], [1, 1])]
        assert (pool.fork_each([]) if use_each else pool.fork_batch([], [])) == []
        pool.sync()
        states.append(([pool.read_table(k) for k in kids], [pool.branch_len(k) for k in kids],
                       pool.read_refcounts(), pool.read_table(b), pool.read_table(a)))
        assert states[-1][0] == [pool.read_table(b), pool.read_table(a)]
        pool.close()
    assert states[0] == states[1]


def test_exhausted_pool_applies_nothing_and_is_sticky():
    pool = Pool(6, 16, 1, 128, torch.bfloat16, max_branches=8, max_blocks_per_branch=8)
    r = pool.new_branch()
    K = torch.randn(1, 24, 1, 128, device="cuda").bfloat16()
    pool.append_kv([r], K, K)
    a, b = pool.fork(r, 2)
    pool.sync()
    before = (pool.read_table(a), pool.read_table(b), pool.read_refcounts(), pool.read_free_stack())
    K2 = torch.randn(2, 40, 1, 128, device="cuda").bfloat16()
    pool.append_kv([a, b], K2, K2)            # needs 2 copies + 4 blocks > 4 free
    assert pool.sync_status() == -2
    with pytest.raises(DendriteError) as e:
        pool.fork(a, 1)
    assert e.value.name == "ENOMEM"
    # device state is exactly as before the failed call (inspection still works;
    # the host length mirror already counted the refused tokens, so the table
    # read covers more entries, and those are still empty)
    ta = pool.read_table(a)
    assert ta[:2] == before[0] and all(x == -1 for x in ta[2:])
    assert pool.read_refcounts() == before[2]
    assert pool.read_free_stack() == before[3]
    pool.close()


def test_host_checked_errors_change_nothing():
    pool = Pool(64, 16, 2, 128, torch.bfloat16, max_branches=4, max_blocks_per_branch=4)
    r = pool.new_branch()
    K = torch.zeros(1, 3, 2, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(DendriteError) as e:
        pool.append_kv([r, r], torch.zeros(2, 3, 2, 128, device="cuda", dtype=torch.bfloat16),
                       torch.zeros(2, 3, 2, 128, device="cuda", dtype=torch.bfloat16))
    assert e.value.name == "EINVAL"
    with pytest.raises(DendriteError) as e:
        pool.fork(r + 1, 1)
    assert e.value.name == "EBADHANDLE"
    with pytest.raises(DendriteError) as e:
        pool.fork(r, 0)
    assert e.value.name == "EINVAL"
    with pytest.raises(DendriteError) as e:
        pool.fork(r, 4)                       # 1 + 4 > 4 handles
    assert e.value.name == "ELIMIT"
    with pytest.raises(DendriteError) as e:   # 5 blocks > 4 per branch
        pool.append_kv([r], torch.zeros(1, 65, 2, 128, device="cuda", dtype=torch.bfloat16),
                       torch.zeros(1, 65, 2, 128, device="cuda", dtype=torch.bfloat16))
    assert e.value.name == "ELIMIT"
    with pytest.raises(DendriteError) as e:   # query longer than the branch
        pool.tree_attn_decode(torch.zeros(1, 1, 2, 128, device="cuda", dtype=torch.bfloat16), [r])
    assert e.value.name == "EINVAL"
    pool.append_kv([r], K, K)
    with pytest.raises(DendriteError) as e:   # n_q_heads not a multiple of n_kv_heads
        pool.tree_attn_decode(torch.zeros(1, 1, 3, 128, device="cuda", dtype=torch.bfloat16), [r])
    assert e.value.name == "EINVAL"
    with pytest.raises(DendriteError):
        pool.append_kv([r], K.float(), K.float())
    pool.free([r])
    with pytest.raises(DendriteError) as e:
        pool.free([r])
    assert e.value.name == "EBADHANDLE"
    pool.sync()
    assert sum(pool.read_refcounts()) == 0
    pool.close()
    for bad in ((64, 8, 2, 128, torch.bfloat16), (64, 16, 2, 64, torch.bfloat16), (64, 16, 2, 48, torch.float32)):
        with pytest.raises(DendriteError) as e:
            Pool(*bad)
        assert e.value.name == "EDTYPE"


def test_fork_chain_cow_stress_small():
    """Chains of d blocks with a half-full tail, forked, each child appends one
    token (copy of the shared half block), then everything is freed."""
    for depth in (1, 3, 10):
        L = W.fork_chain_script(depth)
        ops = [W.Op("new", (0,)), W.Op("append", (0,), L), W.Op("fork", (0,), children=((1, 2, 3, 4),)),
               W.Op("append", (1, 2, 3, 4), 1)]
        w = W.Workload(f"chain{depth}", 8, 32, 128, 16, torch.bfloat16, ops, (1, 2, 3, 4))
        pool = pool_for(w)
        h = run_script(pool, w)
        ref = run_script_pool(w, pool.num_blocks, kv_source=_gpu_kv(w))
        pool.sync()
        pool_state_matches(pool, h, ref)
        pool.free(list(h.values()))
        pool.sync()
        assert pool.read_free_stack() == list(range(pool.num_blocks - 1, -1, -1))
        pool.close()


CAPACITY = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "capacity_cases.json")))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("name", ["exact_fit_copies", "one_short_copies", "exact_fit_last_holder_in_place",
                                  "one_short_in_place"])
def test_capacity_boundary_matches_oracle(name, dtype):
    """Pools sized at exactly an append's block demand, and one block short:
    the exact fit succeeds with the stack emptied, the short one is refused
    (ENOMEM, sticky) with tables, refcounts and stack as before; both
    compared with the hand-derived states and with O2 bit for bit."""
    c = CAPACITY["cases"][name]
    d = 128 if dtype == torch.bfloat16 else 32
    bits = np.uint16 if dtype == torch.bfloat16 else np.uint32
    N = c["num_blocks"]
    pool = Pool(N, 16, 1, d, dtype, max_branches=8, max_blocks_per_branch=8)
    ref = BlockPool(N, 16, 1, d, bits)
    g = torch.Generator(device="cuda").manual_seed(11)
    h = {}
    refused = None
    for i, (kind, branches, *rest) in enumerate(c["script"]):
        if kind == "new":
            h[branches[0]] = pool.new_branch()
            ref.new_branch(branches[0])
        elif kind == "fork":
            for lid, hid in zip(rest[0], pool.fork(h[branches[0]], len(rest[0]))):
                h[lid] = hid
            ref.fork(branches, [rest[0]])
        elif kind == "free":
            pool.free([h[b] for b in branches])
            ref.free(branches)
            for b in branches:
                del h[b]
        elif kind == "append":
            n = rest[0]
            K = torch.randn((len(branches), n, 1, d), generator=g, device="cuda").to(dtype)
            V = torch.randn((len(branches), n, 1, d), generator=g, device="cuda").to(dtype)
            pool.append_kv([h[b] for b in branches], K, V)
            try:
                ref.append(branches, n, bits_of(K), bits_of(V))
            except PoolExhausted:
                refused = i
    assert refused == c.get("exhausted_at_op")
    if refused is None:
        pool.sync()
        for b, tab in c["tables"].items():
            assert pool.read_table(h[int(b)]) == tab
        assert pool.read_refcounts() == c["refcounts"]
        assert pool.read_free_stack() == c["free_stack"]
        for dst, src, fill in c["cow_copies"]:
            kd, vd = pool.read_block(dst)
            ks, vs = pool.read_block(src)
            assert torch.equal(kd[:, :fill], ks[:, :fill]) and torch.equal(vd[:, :fill], vs[:, :fill])
        pool_state_matches(pool, h, ref)
    else:
        assert pool.sync_status() == -2                  # ENOMEM, sticky
        with pytest.raises(DendriteError) as e:
            pool.sync()
        assert e.value.name == "ENOMEM"
        # the refused append applied nothing: tables (up to the old length),
        # refcounts and the stack are the oracle's, which are the derived ones
        for b, tab in c["tables"].items():
            got = pool.read_table(h[int(b)])
            assert got[:len(tab)] == tab and all(x == -1 for x in got[len(tab):])
            assert ref.table[int(b)] == tab
        assert pool.read_refcounts() == c["refcounts"] == ref.refcount.tolist()
        assert pool.read_free_stack() == c["free_stack"] == ref.free_stack()
    pool.close()
