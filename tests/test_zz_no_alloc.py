"""kvq_decode_attention_static: decode attention for callers that cannot
allocate device memory (its workspace is a fixed array inside libkvq.so).

Checked through the C ABI against kvq_decode_attention with a caller
workspace, on two calls in a row, with the attention tolerance the other
tests use.  Kept in its own file, collected last."""
import ctypes

import pytest
import torch

import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, make_kv, make_q
from kvq_testing import assert_attention_close

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
    for call in range(2):
        q = make_q(w, step=call).cuda()
        ref = cache.attention(q)                      # caller-provided workspace
        out = torch.full_like(ref, float("nan"))
        assert fn(cache.handle, q.data_ptr(), w.Hq, out.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert_attention_close(out, ref.double().cpu().numpy(), f"static call {call}")


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
