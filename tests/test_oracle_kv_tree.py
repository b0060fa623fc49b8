"""Pins for the fp64 tree-attention oracle (O1) that do not rely on the oracle
itself: a brute-force naive-copy replay, closed forms, invariants stated by the
Dendrite article (ainews.cool, section 技术深度解析), and planted mistakes that
the pins must catch."""
import math
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import kv_tree
from oracle.kv_tree import KVTree, attention_dense, lse_merge, partial_attention, run_script_tree
from copy_write_forked_gb300 import workloads as W


# ----------------------------------------------------------------------------
# brute force: the "full copy" strategy (every branch owns an explicit copy of
# its whole history; a fork deep-copies it) followed by a whole-matrix softmax
# in long double.  This shares nothing with KVTree's parent-pointer walk.

def naive_copy_replay(w):
    seqs = {}
    for idx, op in enumerate(w.ops):
        if op.kind == "new":
            seqs[op.branches[0]] = ([], [])
        elif op.kind == "fork":
            for p, ch in zip(op.branches, op.children):
                for c in ch:
                    seqs[c] = (list(seqs[p][0]), list(seqs[p][1]))
        elif op.kind == "append":
            if op.n_new == 0:
                continue
            K, V = w.kv(idx)
            for i, b in enumerate(op.branches):
                for t in range(op.n_new):
                    seqs[b][0].append(K[i, t].double().numpy())
                    seqs[b][1].append(V[i, t].double().numpy())
        elif op.kind == "free":
            for b in op.branches:
                del seqs[b]
        elif op.kind == "truncate":
            for b, n in zip(op.branches, op.new_lens):
                seqs[b] = (seqs[b][0][:n], seqs[b][1][:n])
    return seqs


def brute_attention(Q, Krows, Vrows, n_kv):
    """All heads and queries at once: explicit masked score matrix, long double."""
    q_len, n_q, d = Q.shape
    K = np.array(Krows, dtype=np.longdouble)        # [L][n_kv][d]
    V = np.array(Vrows, dtype=np.longdouble)
    L = K.shape[0]
    G = n_q // n_kv
    Qh = np.asarray(Q, dtype=np.longdouble)
    out = np.zeros((q_len, n_q, d), dtype=np.longdouble)
    kv_of_head = np.repeat(np.arange(n_kv), G)      # head h -> kv h // G
    for hq in range(n_q):
        Kh = K[:, kv_of_head[hq], :]                # [L][d]
        Vh = V[:, kv_of_head[hq], :]
        S = Qh[:, hq, :] @ Kh.T / np.sqrt(np.longdouble(d))   # [q_len][L]
        pos = np.arange(L)[None, :]
        lim = (L - q_len + np.arange(q_len))[:, None]
        S = np.where(pos <= lim, S, -np.inf)
        E = np.exp(S - S.max(axis=1, keepdims=True))
        out[:, hq, :] = (E / E.sum(axis=1, keepdims=True)) @ Vh
    return out


def tree_outputs(w):
    tree = run_script_tree(w)
    Q = w.q()
    return {b: tree.attend(b, Q[i]) for i, b in enumerate(w.query)}


def brute_outputs(w):
    seqs = naive_copy_replay(w)
    Q = w.q().double().numpy()
    return {b: brute_attention(Q[i], *seqs[b], w.n_kv_heads) for i, b in enumerate(w.query)}


SCRIPT_SEEDS = list(range(12))


@pytest.mark.parametrize("s", SCRIPT_SEEDS)
def test_tree_equals_dense_attention_on_concatenated_sequence(s):
    q_len = 1 + (s % 3)
    w = W.random_script(s, n_ops=14, max_live=5, max_append=10, n_kv=2, n_q=4, d=8, bs=4,
                        q_len=q_len, seed=100 + s)
    got = tree_outputs(w)
    ref = brute_outputs(w)
    assert got.keys() == ref.keys() and got
    for b in got:
        np.testing.assert_allclose(got[b], ref[b].astype(np.float64), rtol=0, atol=1e-12)


@pytest.mark.parametrize("s", range(8))
def test_tree_with_rollbacks_equals_dense_attention(s):
    w = W.random_script(50 + s, n_ops=18, max_live=5, max_append=10, n_kv=2, n_q=4, d=8, bs=4,
                        q_len=1 + s % 2, seed=300 + s, truncates=True)
    assert any(op.kind == "truncate" for op in w.ops) or s > 5
    got, ref = tree_outputs(w), brute_outputs(w)
    for b in got:
        np.testing.assert_allclose(got[b], ref[b].astype(np.float64), rtol=0, atol=1e-12)


def test_rollback_leaves_children_of_the_old_branch_unchanged():
    rng = np.random.default_rng(11)
    t = KVTree(2, 8)
    t.new_root(0)
    t.append(0, _rand((12, 2, 8), rng), _rand((12, 2, 8), rng))
    t.fork(0, [1])
    Q = _rand((1, 4, 8), rng)
    before = t.attend(1, Q)
    t.truncate(0, 5)
    t.append(0, _rand((9, 2, 8), rng), _rand((9, 2, 8), rng))
    assert np.array_equal(t.attend(1, Q), before)
    assert t.length(0) == 14


def test_tiny_workloads_match_brute_force():
    for v in "abc":
        w = W.tiny_cow(v)
        got, ref = tree_outputs(w), brute_outputs(w)
        for b in got:
            np.testing.assert_allclose(got[b], ref[b].astype(np.float64), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ invariants

def _rand(shape, rng):
    return rng.standard_normal(shape)


def test_fork_leaves_parent_output_unchanged():
    rng = np.random.default_rng(0)
    t = KVTree(2, 8)
    t.new_root(0)
    t.append(0, _rand((11, 2, 8), rng), _rand((11, 2, 8), rng))
    Q = _rand((1, 4, 8), rng)
    before = t.attend(0, Q)
    t.fork(0, [1, 2, 3])
    t.append(1, _rand((5, 2, 8), rng), _rand((5, 2, 8), rng))
    t.append(3, _rand((9, 2, 8), rng), _rand((9, 2, 8), rng))
    after = t.attend(0, Q)
    assert np.array_equal(before, after)


def test_child_without_new_tokens_equals_parent():
    rng = np.random.default_rng(1)
    t = KVTree(2, 8)
    t.new_root(0)
    t.append(0, _rand((13, 2, 8), rng), _rand((13, 2, 8), rng))
    t.fork(0, [1])
    t.append(0, _rand((4, 2, 8), rng), _rand((4, 2, 8), rng))   # parent moves on
    Q = _rand((1, 4, 8), rng)
    t2 = KVTree(2, 8)
    t2.new_root(0)
    K, V = t.materialise(0)
    t2.append(0, K[:13], V[:13])
    assert np.array_equal(t.attend(1, Q), t2.attend(0, Q))


def test_closed_form_constant_values():
    rng = np.random.default_rng(2)
    t = KVTree(2, 8)
    t.new_root(0)
    c = rng.standard_normal((2, 8))
    t.append(0, _rand((9, 2, 8), rng), np.broadcast_to(c, (9, 2, 8)))
    out = t.attend(0, _rand((1, 4, 8), rng))
    np.testing.assert_allclose(out[0, 0], c[0], atol=1e-14)
    np.testing.assert_allclose(out[0, 3], c[1], atol=1e-14)


def test_closed_form_zero_keys_gives_mean_of_visible_values():
    rng = np.random.default_rng(3)
    t = KVTree(1, 8)
    t.new_root(0)
    V = rng.standard_normal((10, 1, 8))
    t.append(0, np.zeros((10, 1, 8)), V)
    out = t.attend(0, _rand((3, 2, 8), rng))        # q_len 3: query j sees 8 + j rows
    for j in range(3):
        np.testing.assert_allclose(out[j, 1], V[:8 + j, 0].mean(axis=0), atol=1e-14)


def test_closed_form_single_visible_token():
    rng = np.random.default_rng(4)
    t = KVTree(2, 8)
    t.new_root(0)
    V = rng.standard_normal((1, 2, 8))
    t.append(0, rng.standard_normal((1, 2, 8)), V)
    out = t.attend(0, _rand((1, 4, 8), rng))
    np.testing.assert_allclose(out[0, 2], V[0, 1], atol=1e-15)


def test_closed_form_scale_is_inverse_sqrt_head_dim():
    # q.k1 = 2, q.k2 = 0, d = 4  ->  scores 1 and 0  ->  weight e / (e + 1)
    t = KVTree(1, 4)
    t.new_root(0)
    K = np.zeros((2, 1, 4)); K[0, 0, 0] = 1.0
    V = np.zeros((2, 1, 4)); V[0, 0, :] = 1.0
    t.append(0, K, V)
    Q = np.zeros((1, 1, 4)); Q[0, 0, 0] = 2.0
    out = t.attend(0, Q)
    np.testing.assert_allclose(out[0, 0], np.full(4, math.e / (math.e + 1)), atol=1e-15)


def test_gqa_head_mapping_groups_consecutive_heads():
    # 2 KV heads with constant values 1 and 2, 4 query heads: heads 0,1 -> 1 and 2,3 -> 2
    t = KVTree(2, 4)
    t.new_root(0)
    V = np.zeros((3, 2, 4)); V[:, 0] = 1.0; V[:, 1] = 2.0
    t.append(0, np.random.default_rng(5).standard_normal((3, 2, 4)), V)
    out = t.attend(0, np.random.default_rng(6).standard_normal((1, 4, 4)))
    np.testing.assert_allclose(out[0, :, 0], [1, 1, 2, 2], atol=1e-14)


def test_lse_merge_of_any_split_equals_unsplit_softmax():
    rng = np.random.default_rng(7)
    for trial in range(20):
        L = int(rng.integers(1, 40))
        d = 8
        q = rng.standard_normal(d)
        K = rng.standard_normal((L, d)) * 3
        V = rng.standard_normal((L, d))
        full = attention_dense(q[None, None], K[:, None], V[:, None])[0, 0]
        cuts = sorted(rng.choice(np.arange(0, L + 1), size=int(rng.integers(0, 5)), replace=True))
        bounds = [0] + list(cuts) + [L]
        parts = [partial_attention(q, K[a:b], V[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        np.testing.assert_allclose(lse_merge(parts), full, atol=1e-13)


def test_last_draft_query_equals_single_decode():
    w = W.spec_verify(requests=2, prefix=21, paths=3, draft=5, n_kv=2, n_q=4, d=8, bs=4,
                      dtype=torch.float32, seed=3)
    tree = run_script_tree(w)
    Q = w.q()
    for i, b in enumerate(w.query):
        full = tree.attend(b, Q[i])
        last = tree.attend(b, Q[i][-1:])
        np.testing.assert_allclose(full[-1], last[0], atol=0)
        # query 0 of the path sees exactly the prefix plus the first draft token
        K, V = tree.materialise(b)
        first = attention_dense(Q[i][:1].double().numpy(), K[:22], V[:22])
        np.testing.assert_allclose(full[0], first[0], atol=0)


# --------------------------------------------------------- planted mistakes

def _mutant(scale=True, gqa="div", vis_shift=0):
    """attention_dense with one planted mistake."""
    def f(Q, K, V):
        q_len, n_q, d = Q.shape
        L, n_kv, _ = K.shape
        G = n_q // n_kv
        out = np.empty((q_len, n_q, d))
        for j in range(q_len):
            vis = max(1, L - q_len + j + 1 + vis_shift)
            for hq in range(n_q):
                kv = hq // G if gqa == "div" else hq % n_kv
                s = K[:vis, kv, :] @ Q[j, hq] / (math.sqrt(d) if scale else 1.0)
                p = np.exp(s - s.max())
                out[j, hq] = (p @ V[:vis, kv, :]) / p.sum()
        return out
    return f


@pytest.mark.parametrize("mutant", [_mutant(scale=False), _mutant(gqa="mod"), _mutant(vis_shift=-1)],
                         ids=["no_scale", "gqa_modulo", "sees_one_less"])
def test_pins_catch_planted_attention_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(kv_tree, "attention_dense", mutant)
    caught = False
    for s in range(4):
        w = W.random_script(s, n_ops=10, max_live=4, max_append=8, n_kv=2, n_q=4, d=8, bs=4,
                            seed=200 + s)
        got, ref = tree_outputs(w), brute_outputs(w)
        if any(not np.allclose(got[b], ref[b].astype(np.float64), atol=1e-9) for b in got):
            caught = True
            break
    assert caught


def test_pins_catch_planted_fork_cut_mistake(monkeypatch):
    # a child that sees the parent's rows appended after the fork
    def bad(self, node):
        empty = np.zeros((0, self.n_kv, self.d))
        pk, pv = (self._materialise(node.parent) if node.parent is not None else (empty, empty))
        ok = np.stack(node.k) if node.k else empty
        ov = np.stack(node.v) if node.v else empty
        return np.concatenate([pk, ok]), np.concatenate([pv, ov])
    monkeypatch.setattr(KVTree, "_materialise", bad)
    rng = np.random.default_rng(9)
    t = KVTree(2, 8)
    t.new_root(0)
    t.append(0, _rand((6, 2, 8), rng), _rand((6, 2, 8), rng))
    t.fork(0, [1])
    t.append(0, _rand((3, 2, 8), rng), _rand((3, 2, 8), rng))
    # pin: a child with no new tokens equals its parent as it was at the fork
    ref = KVTree(2, 8)
    ref.new_root(0)
    K, V = t.materialise(0)
    ref.append(0, K[:6], V[:6])
    Q = _rand((1, 4, 8), rng)
    assert t.attend(1, Q).shape != ref.attend(0, Q).shape or not np.allclose(t.attend(1, Q), ref.attend(0, Q))
