"""The allocation-free attention entry point, through the C-ABI, against the
regular entry point.

Callers such as a serving process whose device memory is already owned by its
own caching allocator, or a latency-critical decode loop that cannot absorb a
cudaMalloc's device synchronisation, use dendrite_tree_attn_decode_noalloc: it
keeps its plan and partial rows in the library's fixed per-device array
instead of allocating.  Its output must match the regular call within the
bf16 tolerance the other tests use, on two calls in a row (the array keeps the
previous call's contents)."""
import ctypes

import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.dendrite import lib
from copy_write_forked_gb300.runner import pool_for, run_script

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def _call(fn, pool, Q, branches, out):
    arr = (ctypes.c_int32 * len(branches))(*branches)
    stream = torch.cuda.current_stream().cuda_stream
    return fn(pool._h, Q.data_ptr(), Q.shape[2], Q.shape[1], ctypes.addressof(arr), len(branches),
              out.data_ptr(), stream)


def test_noalloc_matches_regular_entry_point_on_two_calls():
    w = W.beam(requests=3, prefix=333, width=4, divergent=29)
    pool = pool_for(w)
    h = run_script(pool, w)
    br = [h[b] for b in w.query]
    Q = w.q("cuda")
    ref = torch.empty_like(Q)
    assert _call(lib().dendrite_tree_attn_decode, pool, Q, br, ref) == 0
    for _ in range(2):
        got = torch.full_like(Q, float("nan"))
        assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, got) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        assert (got.float() - ref.float()).abs().max().item() <= TOL
    pool.sync()
    pool.close()


def test_noalloc_fp32_pool_matches_on_two_calls():
    w = W.tiny_cow("b")
    pool = pool_for(w)
    h = run_script(pool, w)
    br = [h[b] for b in w.query]
    Q = w.q("cuda")
    ref = torch.empty_like(Q)
    assert _call(lib().dendrite_tree_attn_decode, pool, Q, br, ref) == 0
    for _ in range(2):
        got = torch.full_like(Q, float("nan"))
        assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, got) == 0
        torch.cuda.synchronize()
        assert (got - ref).abs().max().item() <= 1e-5
    pool.close()


def test_noalloc_rejects_work_beyond_its_scratch():
    # 1024 branches forked from one 16-token root: 32768 output rows, each with
    # at least one partial row of 130 floats -- more than the 16 MiB array
    pool = __import__("copy_write_forked_gb300").Pool(8, 16, 8, 128, torch.bfloat16, max_branches=1100,
                                                       max_blocks_per_branch=4)
    r = pool.new_branch()
    K = torch.randn(1, 16, 8, 128, device="cuda").bfloat16()
    pool.append_kv([r], K, K)
    kids = pool.fork(r, 1024)
    Q = torch.randn(1024, 1, 32, 128, device="cuda").bfloat16()
    out = torch.empty_like(Q)
    assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, kids, out) == -4   # DENDRITE_ELIMIT
    assert _call(lib().dendrite_tree_attn_decode, pool, Q, kids, out) == 0
    pool.sync()
    pool.close()


def test_noalloc_with_tensor_core_units_matches():
    # 40 branches x G 4 = 160 rows per KV head on the prefix: tcgen05 class,
    # whose plan section and partial rows live in the fixed array as well
    w = W.beam(requests=1, prefix=400, width=40, divergent=11)
    pool = pool_for(w)
    h = run_script(pool, w)
    br = [h[b] for b in w.query]
    Q = w.q("cuda")
    ref = torch.empty_like(Q)
    assert _call(lib().dendrite_tree_attn_decode, pool, Q, br, ref) == 0
    assert pool.last_plan_stats()["n_tc_units"] == 8
    for _ in range(2):
        got = torch.full_like(Q, float("nan"))
        assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, got) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        assert (got.float() - ref.float()).abs().max().item() <= TOL
    pool.sync()
    pool.close()


def test_noalloc_calls_allocate_no_device_memory():
    """On a fresh pool that has never run the regular entry point, repeated
    allocation-free calls leave the device's free memory unchanged (after one
    first call, which looks up the array's address and may load the kernels);
    the regular entry point's first call then has to size the pool's
    workspace, so that workspace was still empty."""
    w = W.beam(requests=2, prefix=200, width=3, divergent=21)
    pool = pool_for(w)
    h = run_script(pool, w)
    br = [h[b] for b in w.query]
    Q = w.q("cuda")
    outs = [torch.full_like(Q, float("nan")) for _ in range(4)]
    ref = torch.empty_like(Q)
    pool.sync()
    assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, outs[0]) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for o in outs[1:]:
        assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, o) == 0
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0
    assert _call(lib().dendrite_tree_attn_decode, pool, Q, br, ref) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] < free1
    for o in outs:
        assert (o.float() - ref.float()).abs().max().item() <= TOL
    pool.sync()
    pool.close()


def test_noalloc_refuses_stream_capture():
    """Under an active stream capture the allocation-free call returns
    DENDRITE_EINVAL and enqueues nothing (its plan copy from a pageable host
    buffer cannot be replayed); after the capture it runs as before."""
    w = W.beam(requests=2, prefix=200, width=3, divergent=21)
    pool = pool_for(w)
    h = run_script(pool, w)
    br = [h[b] for b in w.query]
    Q = w.q("cuda")
    out = torch.full_like(Q, float("nan"))
    assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, out) == 0   # first call: address lookup
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        g.capture_begin()
        try:
            rc = _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, out)
        finally:
            g.capture_end()
    assert rc == -1
    again = torch.full_like(Q, float("nan"))
    assert _call(lib().dendrite_tree_attn_decode_noalloc, pool, Q, br, again) == 0
    torch.cuda.synchronize()
    assert torch.equal(again, out)
    pool.sync()
    pool.close()
