"""GPU parity for the attention-sink window (the sequence's first n_sink
tokens kept bf16; PN-Mix sink protection with N_s = 32, InnerQ's
high-precision window): sink, codes, origins, steps and residual
bit-exact against the oracle, decode attention within the tolerance stated
in kvq_testing."""
import numpy as np
import pytest
import torch

import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, make_kv, make_q, make_token
from kvq_testing import (UnitOracles, assert_attention_close, assert_mixed_exports_equal,
                         assert_sink_equal, assert_uniform_exports_equal)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


def run_sink(B, Hkv, n_rep, L, n_sink, appends=0, kb=2, vb=2, mode="uniform", seed=55):
    w = Workload("sink", seed, B=B, Hq=Hkv * n_rep, Hkv=Hkv, T_q=0, r=L, k_bits=kb,
                 v_bits=vb, k_outliers=4, mode=mode, n_bf16=6 if mode == "mixed" else 0,
                 n_uint4=25 if mode == "mixed" else 0)
    K, V = make_kv(w, L)
    imp = None
    if mode == "mixed":
        g = torch.Generator().manual_seed(seed + 1)
        imp = torch.randn(B, Hkv, 128, generator=g).abs()
    cap = 128 * (2 + (L + appends) // 128)
    cache = kvq.KVCache(B, Hkv, cap, kb, vb, mode=mode, n_bf16=w.n_bf16, n_uint4=w.n_uint4,
                        n_sink=n_sink)
    cache.prefill(K.cuda(), V.cuda(), importance=None if imp is None else imp.cuda())
    ref = UnitOracles(range(B * Hkv), Hkv, kb, vb, mode=mode, n_bf16=w.n_bf16,
                      n_uint4=w.n_uint4, n_sink=n_sink)
    ref.prefill(K, V, imp)
    for step in range(appends):
        kn, vn = make_token(w, step)
        cache.append(kn.cuda(), vn.cuda())
        ref.append(kn, vn)
        if cache.lengths()[1] == 128:
            cache.flush(importance=None if imp is None else imp.cuda())
            ref.flush(imp)
    return w, cache, ref


@pytest.mark.parametrize("B,Hkv,n_rep,L,n_sink,appends,kb,vb", [
    (1, 1, 4, 20, 32, 0, 2, 2),            # all tokens are sinks
    (2, 2, 4, 32 + 3 * 128 + 40, 32, 0, 2, 2),
    (1, 2, 8, 32 + 128, 32, 0, 4, 4),      # sink, one group, empty residual
    (2, 1, 2, 10, 32, 60, 2, 2),           # appends fill the sink, then the residual
    (1, 1, 1, 32 + 2 * 128 + 120, 32, 9, 2, 4),   # a flush after the sink
    (1, 3, 4, 300, 1, 0, 4, 2),
    (1, 1, 4, 128 * 2 + 128, 128, 0, 2, 2),       # the largest window
])
def test_sink_uniform_parity(B, Hkv, n_rep, L, n_sink, appends, kb, vb):
    w, cache, ref = run_sink(B, Hkv, n_rep, L, n_sink, appends, kb, vb)
    assert_sink_equal(cache, ref)
    assert_uniform_exports_equal(cache, ref)
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "sink decode")


def test_sink_mixed_parity():
    w, cache, ref = run_sink(2, 2, 8, 32 + 2 * 128 + 50, 32, 0, mode="mixed")
    assert_sink_equal(cache, ref)
    assert_mixed_exports_equal(cache, ref)
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "mixed sink decode")
