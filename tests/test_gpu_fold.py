"""Folded attention plans against the fp64 oracle.

Folding (pool option ``fold_segments``) lets the segments that follow a short
shared segment read its blocks again with their own rows instead of giving
that segment partial rows of its own.  Each case runs the same tree with
folding off (-1), at the default, and with every foldable segment folded
(a percentage far above 100), and compares every output element with the
oracle: 5e-3 for bf16, 1e-5 for fp32."""
import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.runner import pool_for, run_script

from _harness import check_attention

pytestmark = pytest.mark.gpu
TOL_BF16 = 5e-3
TOL_F32 = 1e-5
FOLD_ALL = 1_000_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def run(w, fold, tol, **kw):
    pool = pool_for(w, fold_segments=fold, **kw)
    h = run_script(pool, w)
    out = pool.tree_attn_decode(w.q("cuda"), [h[b] for b in w.query])
    pool.sync()
    st = pool.last_plan_stats()
    check_attention(w, out, list(range(len(w.query))), tol)
    pool.close()
    return out, st


def test_mcts_folded_plans_match_and_drop_partials():
    w = W.mcts(root=256, iters=60, width=4, per_node=32, max_depth=6)
    o_off, st_off = run(w, -1, TOL_BF16)
    o_def, st_def = run(w, 0, TOL_BF16)
    o_all, st_all = run(w, FOLD_ALL, TOL_BF16)
    assert st_def["n_partials"] < st_off["n_partials"]
    assert st_all["n_partials"] <= st_def["n_partials"]
    # folding changes which tiles are streamed (and how often: every row
    # group of a unit streams its tiles) but not the distinct tiles
    assert st_def["unique_tiles"] == st_all["unique_tiles"] == st_off["unique_tiles"]
    for st in (st_off, st_def, st_all):
        assert st["tiles"] >= st["unique_tiles"]
    assert st_def["n_tc_units"] > 0
    for o in (o_def, o_all):
        assert (o.float() - o_off.float()).abs().max().item() <= 2 * TOL_BF16


def test_mcts_folded_on_the_mma_sync_path_only():
    w = W.mcts(root=128, iters=40, width=4, per_node=16, max_depth=8, seed=5)
    _, st = run(w, FOLD_ALL, TOL_BF16, tc_min_rows=-1)
    assert st["n_tc_units"] == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_trees_bf16_fold_everything(seed):
    w = W.random_script(seed, n_ops=40, max_live=10, max_append=60, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=1 + seed % 4, seed=seed)
    run(w, FOLD_ALL, TOL_BF16)


@pytest.mark.parametrize("seed", range(6))
def test_random_trees_fp32_fold_everything(seed):
    w = W.random_script(seed, n_ops=40, max_live=10, max_append=60, n_kv=2, n_q=4, d=64, bs=16,
                        q_len=1 + seed % 3, seed=seed)
    run(w, FOLD_ALL, TOL_F32)


def test_spec_verify_causal_rows_fold_everything():
    # q_len 8: the draft rows see different prefixes of their own blocks
    w = W.spec_verify(requests=2, prefix=300, paths=3, draft=8)
    run(w, FOLD_ALL, TOL_BF16)
