"""Failure detection in the decode kernel without a GPU fault.

Every wait of a decode warp for a record part it staged is bounded.  The
library's failure-detection hook (kvq_set_wait_limit) lowers the bound to
zero polls, so every first wait gives up at once: the warp sets
KVQ_FLAG_TIMEOUT in the cache's status word, still waits (with the full
bound) for its copy in flight, writes empty partials for the rows it leaves
and returns.  The tests check that the call returns, the flag is raised, no
partial of an earlier call enters the merge (a cache with no residual
window: every warp's slice starts with a group, so every row is empty and
comes out NaN), and that after a reset the next call is clean and matches
the oracle.  No wait is made to run forever and no copy is broken."""
import numpy as np
import pytest
import torch

import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, make_kv, make_q
from kvq_testing import UnitOracles, assert_attention_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


@pytest.fixture()
def zero_polls():
    prev = kvq.set_wait_limit(0)
    yield
    kvq.set_wait_limit(-1)
    assert kvq.set_wait_limit(-1) == 1 << 20       # the default is back
    assert prev == 1 << 20


@pytest.mark.parametrize("mode", ["uniform", "mixed"])
def test_wait_gives_up_sets_flag_and_leaves_no_stale_partial(mode):
    w = Workload("timeout", 97, B=2, Hq=8, Hkv=2, T_q=1024, r=0, mode=mode,
                 n_bf16=6 if mode == "mixed" else 0, n_uint4=25 if mode == "mixed" else 0)
    K, V = make_kv(w)
    imp = torch.rand(w.B, w.Hkv, 128, generator=torch.Generator().manual_seed(5)).cuda() \
        if mode == "mixed" else None
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128, mode=mode, n_bf16=w.n_bf16, n_uint4=w.n_uint4)
    cache.prefill(K.cuda(), V.cuda(), importance=imp)
    ws = cache.workspace(w.Hq)
    q0, q1 = make_q(w, step=0).cuda(), make_q(w, step=1).cuda()
    good = cache.attention(q0, workspace=ws)          # fills ws with valid partials
    torch.cuda.synchronize()
    assert cache.status() == 0 and torch.isfinite(good).all()

    prev = kvq.set_wait_limit(0)
    try:
        bad = cache.attention(q1, workspace=ws)        # the call returns
        torch.cuda.synchronize()
        status = cache.status()
    finally:
        kvq.set_wait_limit(prev)
    assert status & kvq.FLAG_TIMEOUT
    # every warp held a group, gave up at its first wait and wrote empty
    # partials: no row is a merge of the earlier call's partials
    assert torch.isnan(bad).all()

    # a reset clears the sticky word; the next call is clean
    cache.reset()
    cache.prefill(K.cuda(), V.cuda(), importance=imp)
    out = cache.attention(q1, workspace=ws)
    torch.cuda.synchronize()
    assert cache.status() == 0
    ref = UnitOracles(range(w.B * w.Hkv), w.Hkv, mode=mode, n_bf16=w.n_bf16, n_uint4=w.n_uint4)
    ref.prefill(K, V, None if imp is None else imp.cpu())
    assert_attention_close(out, ref.attention(make_q(w, step=1)), f"{mode} after reset")


def test_wait_limit_with_residual_rows_returns_and_flags(zero_polls):
    """With a residual window some slices hold no group (they never wait);
    the call still returns, the flag is raised and the rows are finite or
    NaN, never a hang."""
    w = Workload("timeout_res", 98, B=4, Hq=16, Hkv=4, T_q=2048, r=77)
    K, V = make_kv(w)
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128)
    cache.prefill(K.cuda(), V.cuda())
    out = cache.attention(make_q(w).cuda())
    torch.cuda.synchronize()
    assert cache.status() & kvq.FLAG_TIMEOUT
    assert out.shape == (w.B, w.Hq, 128)
    assert not np.isinf(out.cpu().numpy()).any()
