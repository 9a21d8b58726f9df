"""GPU parity for MixKVQ mixed-precision keys: flush/prefill exports
(permutation, raw BF16 tier, UINT4/UINT2 codes, origins, steps) bit-exact
against the oracle, and decode attention over mixed groups within the
tolerance stated in kvq_testing.  Importance I_d always comes from the
oracle (or a seeded generator), never from the GPU path."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as orc
import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import (WORKLOADS, Workload, bf16_bits, make_kv, make_q,
                                              make_query_window, make_token, scaled)
from kvq_testing import UnitOracles, assert_attention_close, assert_mixed_exports_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


def attention_static(cache: kvq.KVCache, q: torch.Tensor) -> torch.Tensor:
    fn = kvq.lib().kvq_decode_attention_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p]
    out = torch.full((q.shape[0], q.shape[1], 128), float("nan"), device=q.device)
    assert fn(cache.handle, q.data_ptr(), q.shape[1], out.data_ptr(),
              torch.cuda.current_stream().cuda_stream) == 0
    return out


def mixed_case(B, Hkv, n_rep, T_q, r, nb, n4, v_bits=2, seed=91) -> Workload:
    return Workload("mixed", seed, B=B, Hq=Hkv * n_rep, Hkv=Hkv, T_q=T_q, r=r, v_bits=v_bits,
                    k_outliers=6, mode="mixed", n_bf16=nb, n_uint4=n4)


def seeded_importance(w: Workload, seed: int) -> torch.Tensor:
    """I_d >= 0 fp32 [B, Hkv, D]: |N(0,1)| with a few large channels and some
    exact ties (ranks then fall back to the channel index)."""
    g = torch.Generator().manual_seed(seed)
    I = torch.randn(w.B, w.Hkv, 128, generator=g).abs()
    I[..., :4] *= 8.0
    I[..., 40:44] = 0.75
    return I.float()


def run_mixed(w: Workload, importance: torch.Tensor, extra_tokens=0, units=None):
    L = w.T - extra_tokens
    K, V = make_kv(w, L)
    units = list(range(w.B * w.Hkv)) if units is None else units
    cap = w.T_q + 128 * (1 + extra_tokens // 128)
    cache = kvq.KVCache(w.B, w.Hkv, cap, 2, w.v_bits, mode="mixed", n_bf16=w.n_bf16,
                        n_uint4=w.n_uint4)
    cache.prefill(K.cuda(), V.cuda(), importance=importance.cuda())
    ref = UnitOracles(units, w.Hkv, 2, w.v_bits, mode="mixed", n_bf16=w.n_bf16,
                      n_uint4=w.n_uint4)
    ref.prefill(K, V, importance)
    for step in range(extra_tokens):
        kn, vn = make_token(w, step)
        cache.append(kn.cuda(), vn.cuda())
        ref.append(kn, vn)
        if cache.lengths()[1] == 128:
            cache.flush(importance=importance.cuda())
            ref.flush(importance)
    return cache, ref


@pytest.mark.parametrize("B,Hkv,L,nb,n4,vb", [
    (1, 1, 128, 6, 25, 2),          # the MixKVQ split: 6 BF16, 25 UINT4, 97 UINT2
    (2, 2, 3 * 128 + 40, 6, 25, 2),
    (1, 2, 2 * 128, 0, 0, 4),       # all UINT2
    (2, 1, 128, 16, 0, 2),          # no UINT4
    (1, 1, 2 * 128 + 5, 0, 128, 2),  # all UINT4: 256 virtual channels
    (1, 1, 128, 128, 0, 4),         # all BF16: no codes
    (1, 3, 128, 3, 125, 2),         # 250 virtual channels, 3 BF16
])
def test_mixed_prefill_exports_bit_exact(B, Hkv, L, nb, n4, vb):
    w = mixed_case(B, Hkv, 1, L - L % 128, L % 128, nb, n4, vb)
    cache, ref = run_mixed(w, seeded_importance(w, 5))
    assert_mixed_exports_equal(cache, ref)


def test_mixed_flush_exports_bit_exact():
    # 2 groups + 120 residual, 8 appends fill the residual, a flush seals it
    w = mixed_case(2, 2, 1, 3 * 128, 3, 6, 25)
    cache, ref = run_mixed(w, seeded_importance(w, 6), extra_tokens=11)
    assert cache.lengths() == (3 * 128, 3)
    assert_mixed_exports_equal(cache, ref)


@pytest.mark.parametrize("B,Hkv,n_rep,T_q,r,nb,n4,vb", [
    (1, 1, 8, 128, 0, 6, 25, 2),
    (2, 2, 8, 640, 37, 6, 25, 2),
    (1, 2, 4, 384, 128, 6, 25, 2),
    (2, 1, 2, 256, 5, 16, 0, 4),
    (1, 2, 1, 512, 64, 0, 128, 2),
    (1, 1, 4, 256, 100, 128, 0, 2),
    (2, 2, 8, 384, 1, 3, 125, 4),
    (1, 1, 8, 0, 77, 6, 25, 2),     # residual only
])
def test_mixed_decode_parity(B, Hkv, n_rep, T_q, r, nb, n4, vb):
    w = mixed_case(B, Hkv, n_rep, T_q, r, nb, n4, vb)
    cache, ref = run_mixed(w, seeded_importance(w, 7))
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "mixed decode")
    assert_attention_close(attention_static(cache, q.cuda()), ref.attention(q), "mixed static")


def test_mixkvq_qwen32b_workload_sampled_units():
    """Qwen-32B-shaped GQA layer (64 query / 8 KV heads), batch 8, 16K
    context, tiers 6/25/97 from a 128-token query window's I_d (oracle)."""
    w = WORKLOADS["mixkvq_qwen32b_16k_b8"]
    qw = make_query_window(w)
    I = np.zeros((w.B, w.Hkv, 128), np.float32)
    for b in range(w.B):
        for h in range(w.Hkv):
            I[b, h] = orc.importance(bf16_bits(qw[b, h * w.n_rep:(h + 1) * w.n_rep]))
    importance = torch.from_numpy(I)
    units = [0, 13, w.B * w.Hkv - 1]
    K, V = make_kv(w, device="cuda")
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128, 2, 2, mode="mixed", n_bf16=6, n_uint4=25)
    cache.prefill(K, V, importance=importance.cuda())
    ref = UnitOracles(units, w.Hkv, 2, 2, mode="mixed", n_bf16=6, n_uint4=25)
    ref.prefill(K.cpu(), V.cpu(), importance)
    del K, V
    q = make_q(w, device="cuda")
    assert_attention_close(cache.attention(q), ref.attention(q.cpu()), w.name)
