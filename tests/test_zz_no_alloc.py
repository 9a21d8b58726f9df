"""kvq_decode_attention_static: decode attention for callers that cannot
allocate device memory (its workspace is a fixed array inside libkvq.so).

Checked through the C ABI against kvq_decode_attention with a caller
workspace, on two calls in a row, with the attention tolerance the other
tests use, and against the CPU oracle; at batches where the split-K split
has to shrink to fit the fixed array; and with the failure-detection wait
limit, where no partial of an earlier call may enter the merge.  Kept in
its own file, collected last."""
import ctypes

import pytest
import torch

import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, make_kv, make_q
from kvq_testing import UnitOracles, assert_attention_close

pytestmark = pytest.mark.gpu

KVQ_ERR_WORKSPACE = 9


def _static_entry():
    _build.build()
    fn = kvq.lib().kvq_decode_attention_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p]
    return fn


def test_static_workspace_matches_caller_workspace_two_calls():
    fn = _static_entry()
    w = Workload("no_alloc", 91, B=4, Hq=32, Hkv=8, T_q=2048, r=45)
    K, V = make_kv(w)
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128)
    cache.prefill(K.cuda(), V.cuda())
    stream = torch.cuda.current_stream().cuda_stream
    orc = UnitOracles((0, 5, 13, 31), w.Hkv)
    orc.prefill(K, V)
    for call in range(2):
        q = make_q(w, step=call).cuda()
        ref = cache.attention(q)                      # caller-provided workspace
        out = torch.full_like(ref, float("nan"))
        assert fn(cache.handle, q.data_ptr(), w.Hq, out.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert_attention_close(out, ref.double().cpu().numpy(), f"static call {call}")
        assert_attention_close(out, orc.attention(make_q(w, step=call)),
                               f"static call {call} vs oracle")


@pytest.mark.parametrize("B,T_q,r", [
    (128, 256, 10),    # 1024 units: three partial slots fit, the split shrinks to 2048 warps
    (252, 128, 5),     # 8064 query rows, just under the limit: two slots, one warp per unit
])
def test_static_workspace_reduced_split_matches(B, T_q, r):
    fn = _static_entry()
    w = Workload("no_alloc_cap", 93, B=B, Hq=32, Hkv=8, T_q=T_q, r=r)
    K, V = make_kv(w, device="cuda")
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128)
    cache.prefill(K, V)
    stream = torch.cuda.current_stream().cuda_stream
    orc = UnitOracles((0, 517, w.B * w.Hkv - 1), w.Hkv)
    orc.prefill(K.cpu(), V.cpu())
    for call in range(2):
        q = make_q(w, step=call, device="cuda")
        ref = cache.attention(q)
        out = torch.full_like(ref, float("nan"))
        assert fn(cache.handle, q.data_ptr(), w.Hq, out.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert_attention_close(out, ref.double().cpu().numpy(), f"B={B} static call {call}")
        assert_attention_close(out, orc.attention(q.cpu()), f"B={B} static call {call} vs oracle")


def test_static_workspace_timeout_leaves_no_stale_partial():
    """A wait that gives up (the failure-detection limit at zero polls) must
    not let the previous call's partials, still in the shared array, into
    the merge: with no residual every warp holds a group, gives up and
    writes empty partials, so every row is NaN and the flag is set."""
    fn = _static_entry()
    w = Workload("no_alloc_timeout", 94, B=2, Hq=8, Hkv=2, T_q=1024, r=0)
    K, V = make_kv(w)
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128)
    cache.prefill(K.cuda(), V.cuda())
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.empty(w.B, w.Hq, 128, dtype=torch.float32, device="cuda")
    assert fn(cache.handle, make_q(w).cuda().data_ptr(), w.Hq, out.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and cache.status() == 0
    prev = kvq.set_wait_limit(0)
    try:
        q1 = make_q(w, step=1).cuda()
        assert fn(cache.handle, q1.data_ptr(), w.Hq, out.data_ptr(), stream) == 0
        torch.cuda.synchronize()
    finally:
        kvq.set_wait_limit(prev)
    assert cache.status() & kvq.FLAG_TIMEOUT
    assert torch.isnan(out).all()


def test_static_workspace_rejects_rows_beyond_the_array():
    fn = _static_entry()
    w = Workload("no_alloc_big", 92, B=2100, Hq=8, Hkv=1, T_q=0, r=1)   # 16800 query rows
    K, V = make_kv(w, L=1)
    cache = kvq.KVCache(w.B, w.Hkv, 128)
    cache.prefill(K.cuda(), V.cuda())
    q = make_q(w).cuda()
    out = torch.zeros(w.B, w.Hq, 128, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert fn(cache.handle, q.data_ptr(), w.Hq, out.data_ptr(), stream) == KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0                # nothing was launched
