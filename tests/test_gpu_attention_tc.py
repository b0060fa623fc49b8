"""The tensor-core (tcgen05) attention path against the fp64 oracle.

Sharing segments read by more than 64 query rows per KV head run on the
tcgen05 kernel (128-row tiles, accumulators in tensor memory).  Each case here
checks that the plan really routes units there, then compares every output
element with the oracle (5e-3 max abs error, bf16 inputs ~ N(0, 1)), and
where useful also with the mma.sync path forced by ``tc_min_rows=-1``."""
import numpy as np
import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.runner import pool_for, run_script

from _harness import check_attention

pytestmark = pytest.mark.gpu
TOL_BF16 = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def run(w, tc_min_rows=0, sample=None):
    pool = pool_for(w, tc_min_rows=tc_min_rows)
    h = run_script(pool, w)
    out = pool.tree_attn_decode(w.q("cuda"), [h[b] for b in w.query])
    pool.sync()
    st = pool.last_plan_stats()
    idx = list(range(len(w.query))) if sample is None else sample
    check_attention(w, out, idx, TOL_BF16)
    pool.close()
    return out, st


def test_wide_fork_256_rows_uses_tc_and_matches():
    # 64 branches x G 4 = 256 rows per KV head on the shared prefix: one
    # two-row-tile unit per head; the stream-K split cuts units into chunks
    w = W.beam(requests=2, prefix=700, width=64, divergent=20)
    out, st = run(w, sample=list(range(0, 128, 5)))
    assert st["n_tc_units"] == 2 * 8 and st["n_tc_ctas"] > 16


def test_rows_between_one_and_two_row_tiles():
    # 40 branches x G 4 = 160 rows: units of 256 rows hold 160 (rt 2, 32 rows padded)
    w = W.beam(requests=1, prefix=333, width=40, divergent=9)
    _, st = run(w)
    assert st["n_tc_units"] == 8


def test_spec_verify_rows_96():
    w = W.spec_verify(requests=3, prefix=500, paths=3, draft=8)
    _, st = run(w)
    assert st["n_tc_units"] == 3 * 8


def test_causal_rows_inside_a_shared_segment():
    # children that appended nothing share the parent's last q_len tokens, so
    # rows of one tcgen05 unit see different prefixes of the same stage
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 203),
           W.Op("fork", (0,), children=(tuple(range(1, 81)),))]
    w = W.Workload("causal_tc", 8, 32, 128, 16, torch.bfloat16, ops, tuple(range(1, 81)), q_len=4, seed=7)
    # 80 members x 4 tokens x G 4 = 1280 rows: 5 units of 256 per head
    _, st = run(w, sample=[0, 17, 39, 40, 63, 79])
    assert st["n_tc_units"] == 5 * 8


def test_mcts_root_row_groups():
    w = W.mcts(root=256, iters=60, width=4, per_node=32, max_depth=6)
    _, st = run(w)
    assert st["n_tc_units"] > 0


def test_tc_and_mma_sync_paths_agree_with_oracle_on_the_same_tree():
    w = W.beam(requests=2, prefix=1000, width=24, divergent=30)
    o_tc, st_tc = run(w)
    o_ms, st_ms = run(w, tc_min_rows=-1)
    assert st_tc["n_tc_units"] > 0 and st_ms["n_tc_units"] == 0
    diff = (o_tc.float() - o_ms.float()).abs().max().item()
    assert diff <= 2 * TOL_BF16


class _Ramp(W.Workload):
    """Keys and queries share a direction u, and the keys' component along u
    grows with the position, so a row's running max rises by far more than 8
    (base 2) across stages: the lazy-rescale path of the tcgen05 kernel runs
    many times.  Values stay N(0, 1)."""

    def kv_one(self, op_index, pos, device="cpu", layer=0):
        k, v = super().kv_one(op_index, pos, device, layer)
        n = k.shape[0]
        start = sum(op.n_new for op in self.ops[:op_index] if op.kind == "append")
        u = torch.ones(self.head_dim, device=device) / self.head_dim ** 0.5
        t = torch.arange(start, start + n, device=device, dtype=torch.float32)
        ramp = (0.19 * t)[:, None, None] * u[None, None, :]
        return (k.float() * 0.3 + ramp).to(self.dtype), v

    def q_one(self, pos, device="cpu"):
        q = super().q_one(pos, device).float()
        u = torch.ones(self.head_dim, device=device) / self.head_dim ** 0.5
        return (0.3 * q + 3.0 * u).to(self.dtype)


def test_running_max_rescales():
    ops = [W.Op("new", (0,)), W.Op("append", (0,), 1100),
           W.Op("fork", (0,), children=(tuple(range(1, 41)),)), W.Op("append", tuple(range(1, 41)), 3)]
    w = _Ramp("ramp", 8, 32, 128, 16, torch.bfloat16, ops, tuple(range(1, 41)), seed=3)
    _, st = run(w, sample=[0, 13, 39])
    assert st["n_tc_units"] == 8
    run(w, tc_min_rows=-1, sample=[0, 13, 39])


def test_repeated_tc_calls_are_deterministic():
    w = W.beam(requests=1, prefix=640, width=48, divergent=7)
    pool = pool_for(w)
    h = run_script(pool, w)
    Q = w.q("cuda")
    br = [h[b] for b in w.query]
    o1 = pool.tree_attn_decode(Q, br).clone()
    o2 = pool.tree_attn_decode(Q, br)
    pool.sync()
    assert pool.last_plan_stats()["n_tc_units"] == 8
    assert torch.equal(o1, o2)
    pool.close()
