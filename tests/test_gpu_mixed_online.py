"""GPU parity for MixKVQ's threshold tiers and online salience window.

Threshold tiers (MixKVQ three-tier strategy: A > tau_BF16 -> BF16,
tau_UINT4 < A -> UINT4, else UINT2) in a key record with room for n_bf16
BF16 and n_uint4 UINT4 channels: every group has its own counts, and a
channel over its tier's room drops one tier.  Exports are compared bit for
bit with the oracle (counts, permutation, raw tier, codes, origins, steps),
decode attention within the tolerance of kvq_testing.

Online window (MixKVQ efficient online salience estimation): each decode
step's query is added to the cache's |q| sums; a flush without an explicit
importance takes I_d from them and starts a new window.  Thresholds are
quantiles of the oracle's own salience values, so the counts vary from
group to group and some groups overflow their room.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, bf16_bits, make_kv, make_q, make_token
from kvq_testing import UnitOracles, assert_attention_close, assert_mixed_exports_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


def case(B, Hkv, n_rep, T_q, r, v_bits=2, seed=311) -> Workload:
    return Workload("mixed_thresh", seed, B=B, Hq=Hkv * n_rep, Hkv=Hkv, T_q=T_q, r=r,
                    v_bits=v_bits, k_outliers=6, mode="mixed", n_bf16=6, n_uint4=25)


def seeded_importance(w: Workload, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    I = torch.randn(w.B, w.Hkv, 128, generator=g).abs()
    I[..., :4] *= 8.0
    I[..., 40:44] = 0.75       # exact ties
    return I.float()


def salience_quantiles(K: torch.Tensor, I: torch.Tensor, n_groups: int, qs) -> list[float]:
    """Quantiles of the oracle's A_d over every (b, kv head, group, channel)."""
    Kb = bf16_bits(K)
    A = []
    for b in range(K.shape[0]):
        for h in range(K.shape[1]):
            for g in range(n_groups):
                S = orc.sensitivity(Kb[b, h, 128 * g:128 * (g + 1)], 2)
                A.append(orc.salience(I[b, h].numpy(), S))
    A = np.concatenate(A)
    return [float(np.float32(np.quantile(A, q))) for q in qs]


def run(w: Workload, I: torch.Tensor, nb, n4, taus, extra_tokens=0):
    L = w.T - extra_tokens
    K, V = make_kv(w, L)
    tau_bf16, tau_uint4 = taus
    cap = w.T_q + 128 * (1 + extra_tokens // 128)
    opts = dict(mode="mixed", n_bf16=nb, n_uint4=n4, tier_mode="threshold",
                tau_bf16=tau_bf16, tau_uint4=tau_uint4)
    cache = kvq.KVCache(w.B, w.Hkv, cap, 2, w.v_bits, **opts)
    cache.prefill(K.cuda(), V.cuda(), importance=I.cuda())
    ref = UnitOracles(range(w.B * w.Hkv), w.Hkv, 2, w.v_bits, **opts)
    ref.prefill(K, V, I)
    for step in range(extra_tokens):
        kn, vn = make_token(w, step)
        cache.append(kn.cuda(), vn.cuda())
        ref.append(kn, vn)
        if cache.lengths()[1] == 128:
            cache.flush(importance=I.cuda())
            ref.flush(I)
    return cache, ref


@pytest.mark.parametrize("B,Hkv,n_rep,T_q,r,nb,n4,qs", [
    (2, 2, 8, 4 * 128, 37, 6, 25, (0.97, 0.70)),    # counts vary, UINT4 often over its room
    (1, 2, 4, 3 * 128, 5, 16, 112, (0.95, 0.50)),   # room for nearly every channel
    (2, 1, 2, 2 * 128, 0, 6, 25, (0.90, 0.99)),     # tau_UINT4 above tau_BF16
    (1, 1, 1, 2 * 128, 64, 0, 0, (0.5, 0.5)),       # no room: all UINT2
])
def test_threshold_tiers_prefill_and_decode(B, Hkv, n_rep, T_q, r, nb, n4, qs):
    w = case(B, Hkv, n_rep, T_q, r)
    I = seeded_importance(w, 17)
    K, _ = make_kv(w, w.T)
    taus = salience_quantiles(K, I, T_q // 128, qs)
    cache, ref = run(w, I, nb, n4, taus)
    assert_mixed_exports_equal(cache, ref)
    counts = cache.export_k_mixed()["counts"].cpu().numpy()
    assert counts[..., 0].max() <= nb and counts[..., 1].max() <= n4
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "threshold decode")


def test_threshold_tiers_flush_path():
    w = case(2, 2, 4, 2 * 128, 3)
    I = seeded_importance(w, 18)
    K, _ = make_kv(w, w.T)
    taus = salience_quantiles(K, I, 2, (0.96, 0.75))
    cache, ref = run(w, I, 6, 25, taus, extra_tokens=140)
    assert cache.lengths() == (2 * 128, 3)   # 119 prefilled + 140 appended
    assert_mixed_exports_equal(cache, ref)
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "threshold flush")


@pytest.mark.parametrize("tier_mode", ["rank", "threshold"])
def test_online_window_flushes(tier_mode):
    """Decode steps observe their query; two flushes take I_d from the
    window (each window starts from zero), one in between is given I_d."""
    w = case(2, 2, 4, 128, 0, seed=313)
    I0 = seeded_importance(w, 19)
    K, V = make_kv(w, w.T)
    taus = salience_quantiles(K, I0, 1, (0.96, 0.75)) if tier_mode == "threshold" else (0.0, 0.0)
    opts = dict(mode="mixed", n_bf16=6, n_uint4=25, tier_mode=tier_mode,
                tau_bf16=taus[0], tau_uint4=taus[1])
    cache = kvq.KVCache(w.B, w.Hkv, 5 * 128, 2, 2, **opts)
    cache.prefill(K.cuda(), V.cuda(), importance=I0.cuda())
    ref = UnitOracles(range(w.B * w.Hkv), w.Hkv, 2, 2, **opts)
    ref.prefill(K, V, I0)
    g = torch.Generator().manual_seed(23)
    for step in range(3 * 128 + 9):
        q = torch.randn(w.B, w.Hq, 128, generator=g)
        q[..., 5] *= 6.0
        q = q.to(torch.bfloat16)
        cache.observe(q.cuda())
        ref.observe(q)
        kn, vn = make_token(w, step)
        cache.append(kn.cuda(), vn.cuda())
        ref.append(kn, vn)
        if cache.lengths()[1] == 128:
            given = step // 128 == 1
            cache.flush(importance=I0.cuda() if given else None)
            ref.flush(I0 if given else None)
    assert cache.lengths() == (4 * 128, 9)
    assert cache.status() == 0
    assert_mixed_exports_equal(cache, ref)
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "online window decode")


def test_online_window_errors():
    w = case(1, 2, 2, 0, 0)
    cache = kvq.KVCache(1, 2, 256, 2, 2, mode="mixed", n_bf16=6, n_uint4=25)
    for step in range(128):
        kn, vn = make_token(w, step)
        cache.append(kn.cuda(), vn.cuda())
    with pytest.raises(kvq.KVQError) as e:      # no query observed in this window
        cache.flush()
    assert e.value.name == "EMPTY"
    q4 = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    q2 = torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    cache.observe(q4)
    with pytest.raises(kvq.KVQError) as e:      # query heads changed within the window
        cache.observe(q2)
    assert e.value.name == "SHAPE"
    with pytest.raises(kvq.KVQError) as e:
        cache.observe(torch.zeros(1, 3, 128, dtype=torch.bfloat16, device="cuda"))
    assert e.value.name == "SHAPE"
    cache.flush()                               # the window holds one step
    assert cache.lengths() == (128, 0)
    cache.observe(q2)                           # a new window may change heads
    uniform = kvq.KVCache(1, 2, 128, 2, 2)
    with pytest.raises(kvq.KVQError) as e:
        uniform.observe(q2)
    assert e.value.name == "MODE"
