"""Pins for the multi-layer form of the block-pool oracle (O2).

The pages describe one attention layer; a model of several layers keeps one
K and V array per layer behind one set of block ids, tables, refcounts and
free stack (every layer of a decoded token lives at the same position).  The
pin: an n-layer pool equals n one-layer pools, each fed that layer's rows,
with identical tables, refcounts and free stacks, over random fork / append /
free / truncate scripts, and the one-layer pool is itself pinned by the
hand-derived states in tests/golden/tiny_cow_states.json.  A planted mistake
(copy-on-write that copies only layer 0) must fail it."""
import json
import os

import numpy as np
import pytest
import torch

from oracle.block_pool import BlockPool, bits_of, run_script_pool
from copy_write_forked_gb300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_cow_states.json")))
N_LAYERS = 3


def single_layer_pool(w, num_blocks, layer):
    """One-layer O2 replay of ``w`` fed the rows of ``layer``."""
    return run_script_pool(w, num_blocks, kv_source=lambda idx: w.kv(idx, layer=layer))


def assert_layers_match(multi, w, num_blocks):
    for l in range(multi.n_layers):
        one = single_layer_pool(w, num_blocks, l)
        assert multi.table == one.table
        assert multi.len == one.len
        assert np.array_equal(multi.refcount, one.refcount)
        assert multi.free_stack() == one.free_stack()
        for b in multi.table:
            ka, va = multi.read_branch_bits(b, layer=l)
            kb, vb = one.read_branch_bits(b)
            assert np.array_equal(ka, kb) and np.array_equal(va, vb), (l, b)


@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_golden_tables_hold_for_every_layer(variant):
    g = GOLDEN["cases"][variant]
    w = W.tiny_cow(variant)
    pool = run_script_pool(w, 64, n_layers=N_LAYERS)
    assert {str(k): v for k, v in pool.table.items()} == g["tables"]
    assert_layers_match(pool, w, 64)


def test_cow_copies_every_layer():
    # tiny case b: both children copy the shared half block 4 into 5 and 7
    w = W.tiny_cow("b")
    pool = run_script_pool(w, 64, n_layers=N_LAYERS)
    for l in range(N_LAYERS):
        for dst in (5, 7):
            assert np.array_equal(pool.KL[l, dst, :, :8], pool.KL[l, 4, :, :8])
            assert np.array_equal(pool.VL[l, dst, :, :8], pool.VL[l, 4, :, :8])
    # layers carry different rows
    assert not np.array_equal(pool.KL[0, 4, :, :8], pool.KL[1, 4, :, :8])


@pytest.mark.parametrize("seed", range(8))
def test_random_scripts_layers_equal_single_layer_pools(seed):
    w = W.random_script(300 + seed, n_ops=40, max_live=6, max_append=30, truncates=seed % 2 == 1, seed=seed)
    nb = w.blocks_upper_bound() + 8
    multi = run_script_pool(w, nb, n_layers=N_LAYERS)
    assert_layers_match(multi, w, nb)


class _Layer0CowOnly(BlockPool):
    """Planted mistake: the copy-on-write copies only layer 0."""

    def append(self, branches, n_new, K_bits, V_bits):
        saved = (self.KL[1:].copy(), self.VL[1:].copy())
        cow = {}
        for b in branches:
            L = self.len[b]
            if L % self.bs and self.refcount[self.table[b][L // self.bs]] > 1:
                cow[b] = L
        super().append(branches, n_new, K_bits, V_bits)
        for b, L in cow.items():
            new = self.table[b][L // self.bs]
            fill = L % self.bs
            self.KL[1:, new, :, :fill] = saved[0][:, new, :, :fill]
            self.VL[1:, new, :, :fill] = saved[1][:, new, :, :fill]


def test_pin_catches_layer0_only_cow(monkeypatch):
    import oracle.block_pool as bp
    monkeypatch.setattr(bp, "BlockPool", _Layer0CowOnly)
    w = W.tiny_cow("b")
    multi = bp.run_script_pool(w, 64, n_layers=N_LAYERS)
    monkeypatch.undo()
    with pytest.raises(AssertionError):
        assert_layers_match(multi, w, 64)
