"""Multi-layer pools through the C-ABI library against the oracle.

A pool of n_layers keeps one K and V pool per layer behind one set of block
ids, tables, refcounts and free stack.  Checked here: the device state (every
layer's bytes) bit-exact against the multi-layer O2 model, attention of every
layer against O1 fed that layer's rows (5e-3, bf16 inputs ~ N(0, 1)), the
split append (append_begin, then append_layer per layer in any order), the
host-checked errors while an append is pending, and plan reuse across the
layers of one step."""
import random

import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.dendrite import DendriteError
from copy_write_forked_gb300.runner import pool_for, run_script
from oracle.block_pool import run_script_pool

from _harness import check_attention, pool_state_matches

pytestmark = pytest.mark.gpu
TOL_BF16 = 5e-3
NL = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def check_all(w, pool, h, n_layers, sample=None):
    ref = run_script_pool(w, pool.num_blocks, n_layers=n_layers, device="cuda")
    pool_state_matches(pool, h, ref, layers=range(n_layers))
    Q = w.q("cuda")
    idx = list(range(len(w.query))) if sample is None else sample
    for l in range(n_layers):
        out = pool.tree_attn_decode(Q, [h[b] for b in w.query], layer=l)
        pool.sync()
        check_attention(w, out, idx, TOL_BF16, layer=l)


@pytest.mark.parametrize("seed", range(4))
def test_random_trees_bulk_append(seed):
    w = W.random_script(400 + seed, n_ops=30, max_live=8, max_append=50, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=1 + seed % 2, seed=seed, truncates=seed % 2 == 1)
    pool = pool_for(w, n_layers=NL)
    h = run_script(pool, w)
    check_all(w, pool, h, NL)
    pool.close()


@pytest.mark.parametrize("seed", range(4))
def test_random_trees_split_append_any_layer_order(seed):
    w = W.random_script(500 + seed, n_ops=30, max_live=8, max_append=50, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=1, seed=seed, truncates=seed % 2 == 0)
    order = list(range(NL))
    random.Random(seed).shuffle(order)
    pool = pool_for(w, n_layers=NL)
    h = run_script(pool, w, split_layers=True, layer_order=order)
    check_all(w, pool, h, NL)
    pool.close()


def test_fp32_layers_tiny_cow():
    w = W.tiny_cow("b")
    pool = pool_for(w, n_layers=2)
    h = run_script(pool, w, split_layers=True, layer_order=[1, 0])
    ref = run_script_pool(w, pool.num_blocks, n_layers=2, device="cuda")
    pool_state_matches(pool, h, ref, layers=(0, 1))
    Q = w.q("cuda")
    for l in range(2):
        out = pool.tree_attn_decode(Q, [h[b] for b in w.query], layer=l)
        pool.sync()
        check_attention(w, out, list(range(len(w.query))), 1e-5, layer=l)
    pool.close()


def test_pending_append_rules():
    w = W.beam(requests=1, prefix=40, width=3, divergent=5, n_kv=2, n_q=8)
    pool = pool_for(w, n_layers=NL, extra_blocks=64)
    h = run_script(pool, w)
    br = [h[b] for b in w.query]
    Q = w.q("cuda")
    out0 = pool.tree_attn_decode(Q, br, layer=1).clone()
    k = torch.randn(len(br), 2, 2, 128, device="cuda").to(torch.bfloat16)
    pool.append_begin(br, 2)
    for bad in (lambda: pool.tree_attn_decode(Q, br, layer=1),
                lambda: pool.free(br[:1]),
                lambda: pool.truncate(br[:1], [3]),
                lambda: pool.append_kv(br, k[None].expand(NL, -1, -1, -1, -1).contiguous(),
                                       k[None].expand(NL, -1, -1, -1, -1).contiguous()),
                lambda: pool.append_begin(br, 1),
                lambda: pool.append_layer(NL, k, k)):
        with pytest.raises(DendriteError) as e:
            bad()
        assert e.value.name == "EINVAL"
    pool.append_layer(1, k, k)
    with pytest.raises(DendriteError):
        pool.append_layer(1, k, k)                 # each layer once
    pool.tree_attn_decode(Q, br, layer=1)          # written layer: allowed
    kids = pool.fork_batch(br[:1], [2])            # forks stay allowed
    pool.append_layer(0, k, k)
    pool.append_layer(2, k, k)
    pool.free(kids[0])                             # no longer pending
    pool.sync()
    assert pool.branch_len(br[0]) == w.lengths()[w.query[0]] + 2
    assert not torch.equal(out0, pool.tree_attn_decode(Q, br, layer=1))
    pool.close()


def test_plan_reused_across_layers_and_tc_path_per_layer():
    # 40 branches x G 4 = 160 rows per KV head on the prefix: tcgen05 class
    w = W.beam(requests=1, prefix=300, width=40, divergent=9)
    pool = pool_for(w, n_layers=NL)
    h = run_script(pool, w)
    Q = w.q("cuda")
    br = [h[b] for b in w.query]
    outs = []
    for l in range(NL):
        outs.append(pool.tree_attn_decode(Q, br, layer=l).clone())
        st = pool.last_plan_stats()
        assert (st["plan_us"] > 0) == (l == 0)
        assert st["n_tc_units"] == 8
    pool.sync()
    for l in range(NL):
        check_attention(w, outs[l], [0, 17, 39], TOL_BF16, layer=l)
    assert not torch.equal(outs[0], outs[1])
    pool.close()
