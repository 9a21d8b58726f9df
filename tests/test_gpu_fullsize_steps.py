"""The benchmarked call at full size: MixKVQ Algorithm 1 decoding through
kvq_decode_step (append, flush when the residual is full, attention) on the
Llama-8B prefill workload (batch 8, 8 KV heads, 32768-token prefill), for
512 steps, so four flushes.  After every flush the new group's exports
(codes, origins, steps, residual) and the step's attention output are
checked against the oracle on sampled (batch row, KV head) units; after the
last one the allocation-free entry point is checked against the oracle too."""
import ctypes

import pytest
import torch

import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import WORKLOADS, make_kv, make_q, make_token
from kvq_testing import UnitOracles, assert_attention_close, assert_uniform_exports_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


def test_decode_steps_across_four_flushes_sampled_units():
    w = WORKLOADS["llama8b_prefill_32k_b8"]
    assert (w.B, w.Hkv, w.T_q, w.steps) == (8, 8, 32768, 512)
    units = [0, 29, 63]
    K, V = make_kv(w, device="cuda")
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128 * 5, w.k_bits, w.v_bits)
    cache.prefill(K, V)
    ref = UnitOracles(units, w.Hkv, w.k_bits, w.v_bits)
    ref.prefill(K, V)
    del K, V
    ws = cache.workspace(w.Hq)
    out = torch.empty(w.B, w.Hq, 128, dtype=torch.float32, device="cuda")
    flushes = 0
    for step in range(w.steps):
        kn, vn = make_token(w, step, device="cuda")
        q = make_q(w, step=step, device="cuda")
        cache.decode_step(kn, vn, q, out=out, workspace=ws)
        ref.append(kn, vn)
        if ref.caches[0].r == 128:          # the step flushed (Alg. 1: before the attention)
            ref.flush()
            flushes += 1
            assert cache.lengths() == (w.T_q + 128 * flushes, 0)
            assert_uniform_exports_equal(cache, ref)
            assert_attention_close(out, ref.attention(q), f"step {step} (flush {flushes})")
    assert flushes == 4 and cache.lengths() == (w.T_q + 512, 0)
    assert cache.status() == 0

    # the allocation-free entry point on the same cache, against the oracle
    fn = kvq.lib().kvq_decode_attention_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] + [ctypes.c_void_p] * 2
    q = make_q(w, step=w.steps, device="cuda")
    out2 = torch.full_like(out, float("nan"))
    assert fn(cache.handle, q.data_ptr(), w.Hq, out2.data_ptr(),
              torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert_attention_close(out2, ref.attention(q), "static entry after four flushes")
