"""Device-side failure handling, exercised without faulting or hanging a GPU.

Every wait in the library's kernels is bounded (about 2 s of %globaltimer).
dendrite_selftest_bounded_wait makes one such wait run out on a barrier that
nothing arrives at: the pool must report DENDRITE_ETIMEOUT at its next sync
and on every later call, and the CUDA context must stay usable for other
pools."""
import ctypes
import time

import pytest
import torch

from copy_write_forked_gb300 import workloads as W
from copy_write_forked_gb300.dendrite import DendriteError, ERRORS, Pool, lib
from copy_write_forked_gb300.runner import pool_for, run_script

from _harness import check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    torch.cuda.set_device(0)


def test_bounded_wait_gives_up_and_poisons_only_its_pool():
    pool = Pool(64, 16, 2, 128, torch.bfloat16, max_branches=8, max_blocks_per_branch=8)
    b = pool.new_branch()
    k = torch.randn(1, 5, 2, 128, device="cuda").to(torch.bfloat16)
    pool.append_kv([b], k, k)
    pool.sync()
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    assert lib().dendrite_selftest_bounded_wait(pool._h, ctypes.c_void_p(stream)) == 0
    st = pool.sync_status()
    waited = time.time() - t0
    assert ERRORS[st] == "ETIMEOUT"
    assert 1.0 < waited < 60.0
    with pytest.raises(DendriteError) as e:   # sticky: later calls report it
        pool.append_kv([b], k, k)
    assert e.value.name == "ETIMEOUT"
    pool.close()
    # the context is fine: another pool works and matches the oracle
    w = W.beam(requests=1, prefix=100, width=2, divergent=7, n_kv=2, n_q=8)
    pool2 = pool_for(w)
    h = run_script(pool2, w)
    out = pool2.tree_attn_decode(w.q("cuda"), [h[x] for x in w.query])
    pool2.sync()
    check_attention(w, out, list(range(len(w.query))), 5e-3)
    pool2.close()
