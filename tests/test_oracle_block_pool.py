"""Pins for the sequential block-pool oracle (O2): hand-derived worked states
(tests/golden/tiny_cow_states.json), invariants, consistency with the logical
tree model O1, and planted mistakes the pins must catch.

Sources: dendrite demo.tape (section "The problem": copy-on-write block table)
and the Dendrite article (ainews.cool, section 技术深度解析: shared prefix stored
once; fork at t shares 0..t-1; memory grows only with divergent tokens)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import block_pool
from oracle.block_pool import BlockPool, PoolExhausted, bits_of, run_script_pool
from oracle.kv_tree import run_script_tree
from copy_write_forked_gb300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_cow_states.json")))
N_TINY = 64


def check_invariants(pool: BlockPool):
    live = pool.table
    # table length matches the branch length
    for b, tab in live.items():
        assert len(tab) == -(-pool.len[b] // pool.bs)
    # sum of refcounts = sum of table lengths
    assert int(pool.refcount.sum()) == sum(len(t) for t in live.values())
    # free count + blocks in use = N, and the free stack holds exactly the unused ids
    used = set(np.nonzero(pool.refcount)[0].tolist())
    free = pool.free_stack()
    assert len(free) + len(used) == pool.N
    assert set(free).isdisjoint(used) and len(set(free)) == len(free)
    # every live entry is referenced; refcount equals the number of holders
    holders = {}
    for tab in live.values():
        for blk in tab:
            holders[blk] = holders.get(blk, 0) + 1
    for blk, n in holders.items():
        assert pool.refcount[blk] == n
    # sharing is prefix-closed below each pair's common full blocks
    items = list(live.items())
    for i in range(len(items)):
        for j in range(i + 1, len(items)):
            a, b = items[i][1], items[j][1]
            n = min(len(a), len(b))
            shared = [k for k in range(n) if a[k] == b[k]]
            if shared:
                assert shared == list(range(len(shared)))


@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_golden_tiny_cow_states(variant):
    g = GOLDEN["cases"][variant]
    w = W.tiny_cow(variant)
    pool = run_script_pool(w, N_TINY)
    assert {str(k): v for k, v in pool.table.items()} == g["tables"]
    assert {str(k): v for k, v in pool.len.items()} == g["lens"]
    rp = g["refcount_prefix"]
    assert pool.refcount[:len(rp)].tolist() == rp
    assert int(pool.refcount[len(rp):].sum()) == 0
    assert pool.used_blocks() == g["used_blocks"]
    for dst, src, fill in g["cow_copies"]:
        assert np.array_equal(pool.K[dst, :, :fill], pool.K[src, :, :fill])
        assert np.array_equal(pool.V[dst, :, :fill], pool.V[src, :, :fill])
    check_invariants(pool)
    pool.free(list(pool.table.keys()))
    assert int(pool.refcount.sum()) == 0
    assert pool.free_stack() == list(range(N_TINY - 1, -1, -1))


def test_golden_truncate_case():
    g = GOLDEN["truncate_case"]
    pool = BlockPool(64, 16, 2, 64, np.uint32)
    rng = np.random.default_rng(0)
    z = lambda n: rng.integers(0, 2**31, size=(1, n, 2, 64), dtype=np.uint32)
    pool.new_branch(0)
    pool.append([0], 20, z(20), z(20))
    pool.fork([0], [[1, 2]])
    pool.append([1], 20, z(20), z(20))
    pool.append([2], 8, z(8), z(8))
    pool.truncate([1, 2], [22, 20])
    pool.free([0])
    pool.append([1], 3, z(3), z(3))
    pool.append([2], 1, z(1), z(1))
    assert {str(k): v for k, v in pool.table.items()} == g["tables"]
    assert {str(k): v for k, v in pool.len.items()} == g["lens"]
    rp = g["refcount_prefix"]
    assert pool.refcount[:len(rp)].tolist() == rp and int(pool.refcount[len(rp):].sum()) == 0
    assert pool.free_stack()[-2:] == g["free_stack_top"]
    assert pool.used_blocks() == g["used_blocks"]
    check_invariants(pool)


@pytest.mark.parametrize("seed", range(15))
def test_invariants_with_rollbacks(seed):
    w = W.random_script(seed, n_ops=40, max_live=8, max_append=12, n_kv=2, n_q=4, d=4, bs=4, truncates=True)
    N = w.blocks_upper_bound() + 3
    for stop in range(1, len(w.ops) + 1):
        check_invariants(run_script_pool(w, N, stop=stop))
    pool = run_script_pool(w, N)
    tree = run_script_tree(w)
    for b in pool.table:
        Kb, _ = pool.read_branch_bits(b)
        Kt, _ = tree.materialise(b)
        assert np.array_equal(Kb.view(np.float32).astype(np.float64), Kt)


def test_sequential_calls_give_same_state_as_one_call():
    # variant c with the two appends issued as separate calls
    w = W.tiny_cow("c")
    ops = list(w.ops)
    last = ops.pop()
    kv = w.kv(len(ops))
    pool = run_script_pool(W.Workload(w.name, 2, 4, 64, 16, torch.float32, ops, (1, 2)), N_TINY)
    K, V = bits_of(kv[0]), bits_of(kv[1])
    pool.append([1], 16, K[0:1], V[0:1])
    pool.append([2], 16, K[1:2], V[1:2])
    ref = run_script_pool(w, N_TINY)
    assert pool.table == ref.table
    assert np.array_equal(pool.refcount, ref.refcount)
    assert np.array_equal(pool.K, ref.K) and np.array_equal(pool.V, ref.V)


@pytest.mark.parametrize("seed", range(25))
def test_invariants_hold_after_every_op_and_free_all_restores(seed):
    w = W.random_script(seed, n_ops=40, max_live=8, max_append=12, n_kv=2, n_q=4, d=4, bs=4)
    N = w.blocks_upper_bound() + 3
    for stop in range(1, len(w.ops) + 1):
        pool = run_script_pool(w, N, stop=stop)
        check_invariants(pool)
    pool.free(list(pool.table.keys()))
    assert int(pool.refcount.sum()) == 0
    assert sorted(pool.free_stack()) == list(range(N))
    if not any(op.kind == "free" for op in w.ops):
        # nothing was released earlier, so one free of everything restores the stack
        assert pool.free_stack() == list(range(N - 1, -1, -1))


@pytest.mark.parametrize("seed", range(10))
def test_block_tables_hold_the_logical_tree_sequences(seed):
    """Reading each branch through its block table gives exactly the sequence
    the logical tree (parent pointers, fork cuts) assigns to it."""
    w = W.random_script(seed, n_ops=30, max_live=6, max_append=11, n_kv=2, n_q=4, d=4, bs=4,
                        dtype=torch.bfloat16)
    pool = run_script_pool(w, w.blocks_upper_bound() + 1)
    tree = run_script_tree(w)
    for b in pool.table:
        Kb, Vb = pool.read_branch_bits(b)
        Kt, Vt = tree.materialise(b)
        got = (Kb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.array_equal(got, Kt)
        got = (Vb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.array_equal(got, Vt)


def test_prefix_stored_once_for_any_fork_width():
    for n in (1, 2, 4, 16, 64):
        pool = BlockPool(512, 16, 1, 4, np.uint32)
        pool.new_branch(0)
        L = 16 * 7 + 5
        pool.append([0], L, np.zeros((1, L, 1, 4), np.uint32), np.zeros((1, L, 1, 4), np.uint32))
        pool.fork([0], [list(range(1, n + 1))])
        assert pool.used_blocks() == -(-L // 16)


def test_memory_grows_only_with_divergent_tokens():
    pool = BlockPool(4096, 16, 1, 4, np.uint32)
    pool.new_branch(0)
    L = 1024
    z = lambda n, m: np.zeros((n, m, 1, 4), np.uint32)
    pool.append([0], L, z(1, L), z(1, L))
    kids = list(range(1, 9))
    pool.fork([0], [kids])
    pool.append(kids, 40, z(8, 40), z(8, 40))
    assert pool.used_blocks() == L // 16 + 8 * 3


def test_exhausted_pool_changes_nothing():
    pool = BlockPool(6, 4, 1, 2, np.uint32)
    pool.new_branch(0)
    pool.append([0], 6, np.ones((1, 6, 1, 2), np.uint32), np.ones((1, 6, 1, 2), np.uint32))
    pool.fork([0], [[1, 2]])
    before = (dict((k, list(v)) for k, v in pool.table.items()), pool.refcount.copy(),
              list(pool.stack), pool.top, pool.K.copy())
    with pytest.raises(PoolExhausted):
        # each child copies the half tail and needs 2 more blocks: 6 > 4 free
        pool.append([1, 2], 8, np.ones((2, 8, 1, 2), np.uint32), np.ones((2, 8, 1, 2), np.uint32))
    assert dict((k, list(v)) for k, v in pool.table.items()) == before[0]
    assert np.array_equal(pool.refcount, before[1])
    assert pool.stack == before[2] and pool.top == before[3]
    assert np.array_equal(pool.K, before[4])


def test_duplicate_branch_in_one_append_is_rejected():
    pool = BlockPool(8, 4, 1, 2, np.uint32)
    pool.new_branch(0)
    with pytest.raises(ValueError):
        pool.append([0, 0], 1, np.zeros((2, 1, 1, 2), np.uint32), np.zeros((2, 1, 1, 2), np.uint32))


# ------------------------------------------------------------ planted mistakes

def test_pins_catch_copy_that_ignores_refcount(monkeypatch):
    orig = BlockPool.append

    def always_copy(self, branches, n_new, K, V):
        # plant: treat every partial tail as shared
        for b in branches:
            L = self.len[b]
            if L % self.bs:
                self.refcount[self.table[b][L // self.bs]] += 1
        try:
            orig(self, branches, n_new, K, V)
        finally:
            pass
    monkeypatch.setattr(BlockPool, "append", always_copy)
    with pytest.raises(AssertionError):
        test_golden_tiny_cow_states("c")


def test_pins_catch_ascending_push(monkeypatch):
    def free_asc(self, branches):
        released = []
        for b in branches:
            for blk in self.table[b]:
                self.refcount[blk] -= 1
                if self.refcount[blk] == 0:
                    released.append(blk)
            del self.table[b]
            del self.len[b]
        for blk in sorted(released):
            self._push(blk)
    monkeypatch.setattr(BlockPool, "free", free_asc)
    with pytest.raises(AssertionError):
        test_golden_tiny_cow_states("a")


def test_pins_catch_fork_without_refcount(monkeypatch):
    # (the planted fork leaves refcounts too low, so the invariant check fails)
    def fork_norc(self, parents, children):
        for p, chs in zip(parents, children):
            for c in chs:
                self.table[c] = list(self.table[p])
                self.len[c] = self.len[p]
    monkeypatch.setattr(BlockPool, "fork", fork_norc)
    with pytest.raises(AssertionError):
        test_invariants_hold_after_every_op_and_free_all_restores(3)


# ------------------------------------------------------- capacity boundary

CAPACITY = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "capacity_cases.json")))


def _replay_capacity_case(name):
    """Replays one hand-derived capacity case on O2 (fp32 payload, 1 KV head,
    head_dim 4); returns the pool and whether the last append was refused."""
    c = CAPACITY["cases"][name]
    pool = BlockPool(c["num_blocks"], CAPACITY["setting"]["block_size"], 1, 4, np.uint32)
    rng = np.random.default_rng(7)
    refused = None
    for i, (kind, branches, *rest) in enumerate(c["script"]):
        if kind == "new":
            pool.new_branch(branches[0])
        elif kind == "fork":
            pool.fork(branches, [rest[0]])
        elif kind == "free":
            pool.free(branches)
        elif kind == "append":
            n = rest[0]
            z = lambda: rng.integers(0, 2**31, size=(len(branches), n, 1, 4), dtype=np.uint32)
            try:
                pool.append(branches, n, z(), z())
            except PoolExhausted:
                refused = i
    return c, pool, refused


@pytest.mark.parametrize("name", ["exact_fit_copies", "one_short_copies", "exact_fit_last_holder_in_place",
                                  "one_short_in_place"])
def test_capacity_boundary_cases(name):
    """An append whose demand equals the free count succeeds and empties the
    stack; one block fewer and it is refused with nothing changed.  The last
    holder of a shared tail whose refcount equals its holders is charged no
    copy (it writes in place)."""
    c, pool, refused = _replay_capacity_case(name)
    assert refused == c.get("exhausted_at_op")
    assert {str(k): v for k, v in pool.table.items()} == c["tables"]
    assert {str(k): v for k, v in pool.len.items()} == c["lens"]
    assert pool.refcount.tolist() == c["refcounts"]
    assert pool.free_stack() == c["free_stack"]
    assert pool.top == len(c["free_stack"])
    for dst, src, fill in c["cow_copies"]:
        assert np.array_equal(pool.K[dst, :, :fill], pool.K[src, :, :fill])
        assert np.array_equal(pool.V[dst, :, :fill], pool.V[src, :, :fill])
    check_invariants(pool)


def _all_capacity_cases():
    for name in CAPACITY["cases"]:
        test_capacity_boundary_cases(name)


def test_pins_catch_refusing_an_exact_fit(monkeypatch):
    # plant: "demand >= free" refuses (demand + 1 > free is the same test)
    orig = BlockPool._demand
    monkeypatch.setattr(BlockPool, "_demand", lambda self, b, n: orig(self, b, n) + 1)
    with pytest.raises(AssertionError):
        _all_capacity_cases()


def test_pins_catch_charging_the_in_place_holder_a_copy(monkeypatch):
    # plant: every holder of a partial tail is charged a copy, the last one included
    def demand_all_copy(self, branches, n_new):
        total = 0
        for b in branches:
            L = self.len[b]
            if L % self.bs and n_new > 0:
                total += 1
            total += -(-(L + n_new) // self.bs) - (-(-L // self.bs))
        return total
    monkeypatch.setattr(BlockPool, "_demand", demand_all_copy)
    with pytest.raises(AssertionError):
        _all_capacity_cases()


def test_pins_catch_a_demand_that_ignores_the_copy(monkeypatch):
    # plant: the copy of a shared tail is not counted, so a one-short call is let through
    def demand_no_copy(self, branches, n_new):
        return sum(-(-(self.len[b] + n_new) // self.bs) - (-(-self.len[b] // self.bs)) for b in branches)
    monkeypatch.setattr(BlockPool, "_demand", demand_no_copy)
    with pytest.raises((AssertionError, IndexError)):
        _all_capacity_cases()
