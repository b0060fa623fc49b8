"""Full-size workloads through the C-ABI library, in the launch configuration
bench.py times, checked against the fp64 oracle on sampled outputs (each
sampled branch is rebuilt in the oracle from its own seeded slices) with the
strict 5e-3 bf16 bound, plus properties that hold at any size."""
import random

import numpy as np
import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.dendrite import Pool
from copy_write_forked_gb300.runner import pool_for, run_script
from oracle.block_pool import BlockPool, bits_of

from _harness import check_attention

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def run_full(w, n_sample, seed=0):
    pool = pool_for(w)
    h = run_script(pool, w)
    Q = w.q("cuda")
    out = pool.tree_attn_decode(Q, [h[b] for b in w.query])
    pool.sync()
    st = pool.last_plan_stats()
    rng = random.Random(seed)
    n = len(w.query)
    sample = sorted(rng.sample(range(n), min(n_sample, n)))
    err = check_attention(w, out, sample, TOL, strict=True)
    assert torch.isfinite(out.float()).all()
    pool.free(list(h.values()))
    pool.sync()
    assert sum(pool.read_refcounts()) == 0
    pool.close()
    return err, st


def test_beam_4096_fork4_256_all_outputs():
    w = W.beam(requests=8, prefix=4096, width=4, divergent=256)
    err, st = run_full(w, n_sample=32)
    assert st["n_segments"] == 8 + 32
    assert st["unique_tiles"] == (8 * 256 + 32 * 16) * 8
    assert st["tiles"] == st["unique_tiles"]


def test_mcts_2048_500_iterations():
    w = W.mcts()
    assert len(w.query) == 1501
    err, st = run_full(w, n_sample=48)
    # 2001 sharing segments (the root's 128 blocks and 2000 nodes of 2 blocks);
    # the plan folds many short ones into the segments that follow them
    assert st["unique_tiles"] == (128 + 2000 * 2) * 8
    assert st["n_segments"] < 2001


def test_spec_verify_8192_3_paths_8_drafts():
    w = W.spec_verify()
    err, st = run_full(w, n_sample=12)


def test_stress_32768_fork64_1024():
    w = W.fork_stress_attention()
    err, st = run_full(w, n_sample=8)
    assert st["unique_tiles"] == (16 * 2048 + 1024 * 64) * 8


def test_fork_stress_100000_forks_with_cow_appends():
    """Chains of 1..500 blocks with a half-full tail; 5000 batches, each forks
    every chain 4 ways (20 forks), appends one token to every child (a copy of
    the shared half block) and frees the children.  Bit-exact against O2 at
    checkpoints; the pool returns to its post-setup state."""
    depths = (1, 10, 50, 100, 500)
    N = sum(depths) + 5 + 64
    pool = Pool(N, 16, 8, 128, torch.bfloat16, max_branches=64, max_blocks_per_branch=512)
    ref = BlockPool(N, 16, 8, 128, np.uint16)
    roots = []
    for i, d in enumerate(depths):
        r = pool.new_branch()
        roots.append(r)
        ref.new_branch(r)
        L = W.fork_chain_script(d)
        g = torch.Generator(device="cuda").manual_seed(W.seed_of("chain", d))
        K = torch.randn(1, L, 8, 128, generator=g, device="cuda").bfloat16()
        V = torch.randn(1, L, 8, 128, generator=g, device="cuda").bfloat16()
        pool.append_kv([r], K, V)
        ref.append([r], L, bits_of(K), bits_of(V))
    pool.sync()
    stack0 = pool.read_free_stack()
    assert stack0 == ref.free_stack()
    g = torch.Generator(device="cuda").manual_seed(W.seed_of("chain", "append"))
    Kt = torch.randn(20, 1, 8, 128, generator=g, device="cuda").bfloat16()
    Vt = torch.randn(20, 1, 8, 128, generator=g, device="cuda").bfloat16()
    Kb, Vb = bits_of(Kt), bits_of(Vt)
    forks = 0
    for batch in range(5000):
        kids = pool.fork_batch(roots, [4] * len(roots))
        flat = [c for ks in kids for c in ks]
        forks += len(flat)
        pool.append_kv(flat, Kt, Vt)
        ref.fork(roots, kids)
        ref.append(flat, 1, Kb, Vb)
        if batch % 1000 == 0 or batch == 4999:
            pool.sync()
            for c in flat[::3]:
                assert pool.read_table(c) == ref.table[c]
            assert pool.read_refcounts() == ref.refcount.tolist()
            assert pool.read_free_stack() == ref.free_stack()
            # the copied half blocks hold the parent's 8 valid slots
            for c, r in zip(flat[::4], roots):
                blk, src = ref.table[c][-1], ref.table[r][-1]
                k, _ = pool.read_block(blk)
                ks, _ = pool.read_block(src)
                assert torch.equal(k[:, :8], ks[:, :8])
        pool.free(flat)
        ref.free(flat)
    pool.sync()
    assert forks == 100000
    assert pool.read_free_stack() == stack0
    assert pool.read_refcounts() == ref.refcount.tolist()
    pool.close()
