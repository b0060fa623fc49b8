"""Tree decode attention through the C-ABI library against the fp64 oracle,
element by element: fp32 pools within 1e-5, bf16 pools within 5e-3 (max abs
error; inputs ~ N(0, 1), fp32 accumulation, output rounded to bf16)."""
import numpy as np
import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.dendrite import Pool
from copy_write_forked_gb300.runner import pool_for, run_script

from _harness import check_attention

pytestmark = pytest.mark.gpu
TOL_BF16 = 5e-3
TOL_F32 = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def run_and_check(w, tol, sample=None, **opts):
    pool = pool_for(w, **opts)
    h = run_script(pool, w)
    Q = w.q("cuda")
    out = pool.tree_attn_decode(Q, [h[b] for b in w.query])
    pool.sync()
    idx = list(range(len(w.query))) if sample is None else sample
    err = check_attention(w, out, idx, tol)
    stats = pool.last_plan_stats()
    pool.close()
    return err, stats


@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_tiny_fp32(variant):
    run_and_check(W.tiny_cow(variant), TOL_F32)


@pytest.mark.parametrize("seed", range(12))
def test_random_trees_fp32(seed):
    q_len = 1 + seed % 3
    w = W.random_script(seed, n_ops=30, max_live=8, max_append=70, n_kv=2, n_q=4, d=64, bs=16,
                        q_len=q_len, seed=seed)
    run_and_check(w, TOL_F32)


@pytest.mark.parametrize("seed", range(12))
def test_random_trees_bf16(seed):
    q_len = 1 + seed % 4
    w = W.random_script(seed, n_ops=30, max_live=8, max_append=90, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=q_len, seed=seed)
    run_and_check(w, TOL_BF16)


def test_beam_small_ragged():
    # ragged prefix and leaves: partial blocks at the fork point and at every tail
    w = W.beam(requests=3, prefix=211, width=4, divergent=37)
    err, st = run_and_check(w, TOL_BF16, pack_segments=-1)
    assert st["n_segments"] == 3 + 12
    # packed (the default): each prefix takes its four leaves' tiles
    err, st = run_and_check(w, TOL_BF16)
    assert st["n_segments"] == 3


def test_wide_fork_spans_row_groups():
    # 20 branches x G=4 = 80 rows per KV head: row groups of 64 and 16
    w = W.beam(requests=2, prefix=300, width=20, divergent=5)
    run_and_check(w, TOL_BF16)


def test_gqa_group_8_and_group_1():
    for n_kv, n_q in ((2, 16), (8, 8)):
        w = W.beam(requests=2, prefix=150, width=3, divergent=20, n_kv=n_kv, n_q=n_q)
        run_and_check(w, TOL_BF16)


def grouped_merge_runs(w):
    """Whether the attention call merges a GQA group's heads together: a
    group of 1, 2 or a multiple of 4 heads, and at least 16 grouped warps per
    SM (smaller merges keep one row per warp)."""
    G = w.n_q_heads // w.n_kv_heads
    ng = 4 if G % 4 == 0 else (G if G in (1, 2) else 0)
    n_out = len(w.query) * w.q_len * w.n_q_heads
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return w.head_dim == 128 and ng > 0 and n_out // ng >= 16 * sms


@pytest.mark.parametrize("n_kv, n_q", [(8, 32), (8, 16), (8, 8), (2, 32), (4, 24)])
def test_grouped_merge_bf16(n_kv, n_q):
    # 48 branches x 8 draft tokens: GQA groups of 4, 2, 1, 16 and 6 heads
    # (the last one merges a row per warp)
    w = W.spec_verify(requests=16, prefix=200, paths=3, draft=8, n_kv=n_kv, n_q=n_q, seed=n_q)
    assert grouped_merge_runs(w) == (n_q // n_kv != 6)
    run_and_check(w, TOL_BF16)


def test_grouped_merge_fp32_head_dim_128():
    w = W.spec_verify(requests=16, prefix=120, paths=3, draft=8, n_kv=8, n_q=32, dtype=torch.float32, seed=3)
    assert grouped_merge_runs(w)
    run_and_check(w, TOL_F32)


@pytest.mark.parametrize("n_kv, n_q", [(2, 6), (1, 12)])
def test_small_merges_odd_groups(n_kv, n_q):
    w = W.random_script(7 + n_q, n_ops=30, max_live=8, max_append=60, n_kv=n_kv, n_q=n_q, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=2, seed=n_q)
    run_and_check(w, TOL_BF16)


@pytest.mark.parametrize("make", [lambda: W.beam(requests=2, prefix=100, width=3, divergent=5),
                                  lambda: W.spec_verify(requests=2, prefix=100, paths=3, draft=8)])
def test_appends_within_blocks_refresh_the_plan(make):
    """A decode loop without forks: every step appends one token to each
    queried branch and attends again.  While no queried branch reaches a new
    block the cached plan only has its lengths refreshed; on the step that
    crosses a block boundary each branch's own last segment is lengthened.
    Every step matches the oracle."""
    base = make()
    extra = [W.Op("append", tuple(base.query), 1) for _ in range(10)]
    w_full = W.Workload(base.name + "_decode", base.n_kv_heads, base.n_q_heads, base.head_dim, base.block_size,
                        base.dtype, list(base.ops) + extra, base.query, base.q_len, base.seed)
    pool = pool_for(w_full)
    h = run_script(pool, base)
    br = [h[b] for b in base.query]
    Q = base.q("cuda")
    pool.tree_attn_decode(Q, br)
    assert pool.last_plan_stats()["refreshed"] == 0
    lens = {b: l for b, l in base.lengths().items()}
    seen = set()
    for k in range(len(extra)):
        idx = len(base.ops) + k
        blocks_before = {b: -(-lens[b] // 16) for b in base.query}
        K, V = w_full.kv(idx, "cuda")
        pool.append_kv(br, K, V)
        for b in base.query:
            lens[b] += 1
        out = pool.tree_attn_decode(Q, br)
        pool.sync()
        st = pool.last_plan_stats()
        crossed = any(-(-lens[b] // 16) != blocks_before[b] for b in base.query)
        assert st["refreshed"] == (2 if crossed else 1), (k, crossed)
        seen.add(st["refreshed"])
        w_k = W.Workload(w_full.name, w_full.n_kv_heads, w_full.n_q_heads, w_full.head_dim, w_full.block_size,
                         w_full.dtype, w_full.ops[:idx + 1], w_full.query, w_full.q_len, w_full.seed)
        check_attention(w_k, out, list(range(len(base.query))), TOL_BF16)
    assert seen == {1, 2}
    pool.close()


def test_mcts_small():
    w = W.mcts(root=256, iters=60, width=4, per_node=32, max_depth=6)
    run_and_check(w, TOL_BF16)


def test_spec_verify_small_causal():
    w = W.spec_verify(requests=3, prefix=500, paths=3, draft=8)
    run_and_check(w, TOL_BF16)


def test_child_with_no_new_tokens_and_single_token_branch():
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 1), W.Op("new", (1,)), W.Op("append", (1,), 45),
           W.Op("fork", (1,), children=((2, 3),)), W.Op("append", (3,), 2)]
    w = W.Workload("edge", 2, 4, 128, 16, torch.bfloat16, ops, (0, 1, 2, 3))
    run_and_check(w, TOL_BF16)


def test_repeated_calls_reuse_the_plan_and_agree():
    w = W.beam(requests=2, prefix=333, width=4, divergent=21)
    pool = pool_for(w)
    h = run_script(pool, w)
    Q = w.q("cuda")
    br = [h[b] for b in w.query]
    o1 = pool.tree_attn_decode(Q, br).clone()
    assert pool.last_plan_stats()["plan_us"] > 0
    o2 = pool.tree_attn_decode(Q, br)
    assert pool.last_plan_stats()["plan_us"] == 0
    assert torch.equal(o1, o2)
    pool.close()


@pytest.mark.parametrize("seed", range(6))
def test_random_trees_with_rollbacks_bf16(seed):
    w = W.random_script(200 + seed, n_ops=30, max_live=8, max_append=90, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=1 + seed % 2, seed=seed, truncates=True)
    run_and_check(w, TOL_BF16)


def test_speculative_accept_and_rollback():
    """Verify 3 draft paths of 8 tokens, keep 5 tokens of path 1, drop the others,
    then decode one more token on the winner."""
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 700), W.Op("fork", (0,), children=((1, 2, 3),)),
           W.Op("append", (1, 2, 3), 8), W.Op("truncate", (2,), new_lens=(705,)), W.Op("free", (1, 3)),
           W.Op("append", (2,), 1)]
    w = W.Workload("accept", 8, 32, 128, 16, torch.bfloat16, ops, (0, 2), 1)
    run_and_check(w, TOL_BF16)


def test_attention_after_free_of_shared_parent():
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 100), W.Op("fork", (0,), children=((1, 2),)),
           W.Op("free", (0,)), W.Op("append", (1, 2), 30)]
    w = W.Workload("orphans", 2, 4, 128, 16, torch.bfloat16, ops, (1, 2))
    run_and_check(w, TOL_BF16)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("tc_min_rows", [0, -1])
def test_random_trees_packed_everywhere_bf16(seed, tc_min_rows):
    """Packing forced wherever the planner allows it (pack_segments far above
    100 percent): packed units read their followers' tiles with per-tile row
    masks, on the mma.sync kernel and (with enough rows) on the tcgen05
    kernel; q_len 1..3 puts a member's causal limits inside its own tiles."""
    q_len = 1 + seed % 3
    w = W.random_script(seed, n_ops=40, max_live=12, max_append=90, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=q_len, seed=seed)
    pool = pool_for(w, pack_segments=1_000_000, tc_min_rows=tc_min_rows if tc_min_rows else 8)
    h = run_script(pool, w)
    out = pool.tree_attn_decode(w.q("cuda"), [h[b] for b in w.query])
    pool.sync()
    check_attention(w, out, list(range(len(w.query))), TOL_BF16)
    pool.close()


@pytest.mark.parametrize("make", [lambda: W.spec_verify(requests=3, prefix=700, paths=3, draft=8),
                                  lambda: W.beam(requests=3, prefix=500, width=4, divergent=40),
                                  lambda: W.mcts(root=300, iters=60, width=4, per_node=24)],
                         ids=["spec_verify", "beam", "mcts"])
def test_packed_and_unpacked_plans_agree_with_the_oracle(make):
    """A plan packed as far as the planner allows reads fewer units than the
    plan with packing off, and both (and the default plan) match the oracle."""
    w = make()
    units = []
    for pack in (1_000_000, -1, 0):
        pool = pool_for(w, pack_segments=pack)
        h = run_script(pool, w)
        out = pool.tree_attn_decode(w.q("cuda"), [h[b] for b in w.query])
        pool.sync()
        units.append(pool.last_plan_stats()["n_units"])
        check_attention(w, out, list(range(len(w.query))), TOL_BF16)
        pool.close()
    assert units[0] < units[1]
