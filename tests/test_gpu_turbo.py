"""Compressed KV blocks (TurboQuant: PolarQuant + QJL; dendrite demo.tape,
section "TurboQuant") through the C-ABI library against the oracle O3: every
stored key and value record bit for bit (fresh encodes and copy-on-write
copies alike), tables and refcounts against O2, and tree decode attention
over the compressed rows within 5e-3 (plus half a bf16 ulp of the output)."""
import random

import numpy as np
import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.runner import pool_for, run_script
from oracle import turbo_quant as T
from oracle.block_pool import run_script_pool

from _harness import half_ulp_bf16, oracle_tree, pool_state_matches

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def _codec(seed=0):
    signs, S = W.turbo_codec(seed)
    return signs, S, signs.numpy().astype(np.float64), S.numpy()


def _expected_records(w, ids, signs, S):
    """Oracle records of every position of each branch in ``ids``: [len][n_kv][96] / [64]."""
    tree = oracle_tree(w, ids, "cuda")
    out = {}
    for b in ids:
        K, V = tree.materialise(b)
        keys = T.pack_key(*T.encode_key(K.astype(np.float32), signs, S))
        vals = T.pack_value(*T.encode_value(V.astype(np.float32), signs))
        out[b] = (keys, vals)
    return out, tree


def _check_records(pool, h, w, ids, signs, S):
    exp, tree = _expected_records(w, ids, signs, S)
    for b in ids:
        tab = pool.read_table(h[b])
        keys, vals = exp[b]
        for pos in range(len(keys)):
            kb, vb = pool.read_block(tab[pos // 16])
            assert np.array_equal(kb[:, pos % 16].numpy(), keys[pos]), ("key record", b, pos)
            assert np.array_equal(vb[:, pos % 16].numpy(), vals[pos]), ("value record", b, pos)
    return exp, tree


@pytest.mark.parametrize("seed", range(6))
def test_records_and_tables_match_the_oracle(seed):
    w = W.random_script(200 + seed, n_ops=24, max_live=6, max_append=40, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16)
    ts, tS, signs, S = _codec(seed)
    pool = pool_for(w, turbo=(ts, tS))
    h = run_script(pool, w)
    pool.sync()
    ref = run_script_pool(w, pool.num_blocks, kv_source=lambda idx: w.kv(idx, "cuda"))
    pool_state_matches(pool, h, ref, check_bytes=False)
    _check_records(pool, h, w, list(ref.table.keys()), signs, S)
    pool.close()


def test_copy_on_write_copies_records():
    # tiny CoW case b, bf16 and head_dim 128: both children copy the shared half block
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 64), W.Op("append", (0,), 8),
           W.Op("fork", (0,), children=((1, 2),)), W.Op("append", (1, 2), 16)]
    w = W.Workload("tiny_b_turbo", 2, 4, 128, 16, torch.bfloat16, ops, (1, 2))
    ts, tS, signs, S = _codec(1)
    pool = pool_for(w, turbo=(ts, tS))
    h = run_script(pool, w)
    pool.sync()
    t0, t1, t2 = pool.read_table(h[0]), pool.read_table(h[1]), pool.read_table(h[2])
    assert t1[4] != t0[4] and t2[4] != t0[4]
    k0, v0 = pool.read_block(t0[4])
    for t in (t1, t2):
        k, v = pool.read_block(t[4])
        assert torch.equal(k[:, :8], k0[:, :8]) and torch.equal(v[:, :8], v0[:, :8])
    _check_records(pool, h, w, [0, 1, 2], signs, S)
    pool.close()


def _check_attention(pool, h, w, signs, S, sample=None):
    Q = w.q("cuda")
    out = pool.tree_attn_decode(Q, [h[b] for b in w.query])
    pool.sync()
    idx = range(len(w.query)) if sample is None else sample
    ids = [w.query[i] for i in idx]
    exp, tree = _expected_records(w, ids, signs, S)
    worst = 0.0
    for i in idx:
        keys, vals = exp[w.query[i]]
        ref = T.attention_compressed(Q[i].double().cpu().numpy(), keys, vals, signs, S, w.n_kv_heads)
        got = out[i].double().cpu().numpy()
        err = np.abs(got - ref)
        worst = max(worst, float(err.max()))
        assert np.isfinite(got).all()
        assert (err <= TOL + half_ulp_bf16(ref)).all(), (i, float(err.max()))
    return worst


@pytest.mark.parametrize("seed", range(6))
def test_attention_over_compressed_rows_matches_the_oracle(seed):
    q_len = 1 + seed % 3
    w = W.random_script(300 + seed, n_ops=24, max_live=6, max_append=60, n_kv=2, n_q=8, d=128, bs=16,
                        dtype=torch.bfloat16, q_len=q_len, seed=seed)
    ts, tS, signs, S = _codec(seed)
    pool = pool_for(w, turbo=(ts, tS))
    h = run_script(pool, w)
    _check_attention(pool, h, w, signs, S)
    pool.close()


def test_beam_shaped_tree_over_compressed_rows():
    """Shared prefixes read by 4 branches (16 rows per KV head), GQA 4, 8 KV heads."""
    w = W.beam(requests=2, prefix=200, width=4, divergent=37)
    ts, tS, signs, S = _codec(7)
    pool = pool_for(w, turbo=(ts, tS))
    h = run_script(pool, w)
    _check_attention(pool, h, w, signs, S, sample=[0, 3, 5])
    pool.close()


@pytest.mark.parametrize("prefix,divergent", [(1500, 300), (4096, 16)])
def test_long_shared_prefix_over_compressed_rows(prefix, divergent):
    """Long prefixes: every warp of a CTA takes many tiles of a unit (the
    per-warp softmax states, the running value scale and the end-of-chunk
    merge of four warps all carry weight)."""
    w = W.beam(requests=2, prefix=prefix, width=4, divergent=divergent)
    ts, tS, signs, S = _codec(11)
    pool = pool_for(w, turbo=(ts, tS))
    h = run_script(pool, w)
    _check_attention(pool, h, w, signs, S, sample=[0, 2, 5, 7])
    pool.close()


@pytest.mark.parametrize("width,q_len", [(16, 1), (6, 2), (3, 3)])
def test_wide_units_share_each_tiles_decode(width, q_len):
    """More than 16 query rows per KV head on a shared prefix (16 x G 4 = 64,
    6 x 2 x 4 = 48 and 3 x 3 x 4 = 36 rows): units of up to 64 rows whose
    tiles the CTA decodes once for all its warps, each warp running 16 of the
    rows (a warp past the unit's rows only decodes); causal queries for
    q_len > 1."""
    if q_len == 1:
        w = W.beam(requests=2, prefix=700, width=width, divergent=20)
    else:
        w = W.spec_verify(requests=2, prefix=500, paths=width, draft=q_len)
    ts, tS, signs, S = _codec(13 + width)
    pool = pool_for(w, turbo=(ts, tS))
    h = run_script(pool, w)
    _check_attention(pool, h, w, signs, S, sample=[0, len(w.query) // 2, len(w.query) - 1])
    pool.close()


def test_multilayer_split_append_encodes_every_layer():
    w = W.beam(requests=1, prefix=40, width=2, divergent=9, n_kv=2, n_q=4)
    ts, tS, signs, S = _codec(3)
    pool = pool_for(w, turbo=(ts, tS), n_layers=2)
    h = run_script(pool, w, split_layers=True, layer_order=[1, 0])
    pool.sync()
    for layer in (0, 1):
        tree = oracle_tree(w, w.query, "cuda", layer)
        for b in w.query:
            K, V = tree.materialise(b)
            keys = T.pack_key(*T.encode_key(K.astype(np.float32), signs, S))
            vals = T.pack_value(*T.encode_value(V.astype(np.float32), signs))
            tab = pool.read_table(h[b])
            for pos in range(len(keys)):
                kb, vb = pool.read_block(tab[pos // 16], layer=layer)
                assert np.array_equal(kb[:, pos % 16].numpy(), keys[pos]), (layer, b, pos)
                assert np.array_equal(vb[:, pos % 16].numpy(), vals[pos]), (layer, b, pos)
    pool.close()


def test_compressed_pool_rejects_the_allocation_free_call():
    from copy_write_forked_gb300.dendrite import DendriteError
    w = W.beam(requests=1, prefix=20, width=2, divergent=3)
    ts, tS, _, _ = _codec(0)
    pool = pool_for(w, turbo=(ts, tS))
    h = run_script(pool, w)
    Q = w.q("cuda")
    with pytest.raises(DendriteError) as e:
        pool.tree_attn_decode_noalloc(Q, [h[b] for b in w.query], torch.empty_like(Q))
    assert e.value.name == "EDTYPE"
    pool.close()
