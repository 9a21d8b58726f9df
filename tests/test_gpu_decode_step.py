"""kvq_decode_step (append, flush when the residual is full, attention in
one call) against the three separate calls on an identical cache: outputs
bit for bit equal at every step, including the steps that fall back to the
separate calls (a flush, the attention-sink window filling), then the
caches' exports equal and the last output within tolerance of the oracle."""
import pytest
import torch

import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, make_kv, make_q, make_token
from kvq_testing import UnitOracles, assert_attention_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


@pytest.mark.parametrize("B,Hkv,n_rep,L,steps,kb,vb,n_sink,mode", [
    (2, 2, 4, 2 * 128 + 120, 20, 2, 2, 0, "uniform"),   # a flush at the 8th step
    (1, 3, 2, 128 + 5, 12, 4, 4, 0, "uniform"),
    (1, 2, 8, 3, 40, 2, 2, 8, "uniform"),                # the sink fills first
    (2, 1, 4, 128 + 30, 10, 2, 2, 0, "mixed"),           # mixed keys, no flush
])
def test_decode_step_equals_separate_calls(B, Hkv, n_rep, L, steps, kb, vb, n_sink, mode):
    w = Workload("step", 91, B=B, Hq=Hkv * n_rep, Hkv=Hkv, T_q=0, r=L, k_bits=kb, v_bits=vb,
                 k_outliers=4, mode=mode, n_bf16=6 if mode == "mixed" else 0,
                 n_uint4=25 if mode == "mixed" else 0)
    K, V = make_kv(w, L)
    imp = None
    if mode == "mixed":
        g = torch.Generator().manual_seed(17)
        imp = torch.randn(B, Hkv, 128, generator=g).abs().cuda()
    cap = 128 * (3 + (L + steps) // 128)

    def fresh():
        c = kvq.KVCache(B, Hkv, cap, kb, vb, mode=mode, n_bf16=w.n_bf16, n_uint4=w.n_uint4,
                        n_sink=n_sink)
        c.prefill(K.cuda(), V.cuda(), importance=imp)
        return c

    fused, split = fresh(), fresh()
    ws_f, ws_s = fused.workspace(w.Hq), split.workspace(w.Hq)
    ref = UnitOracles(range(B * Hkv), Hkv, kb, vb, mode=mode, n_bf16=w.n_bf16,
                      n_uint4=w.n_uint4, n_sink=n_sink)
    ref.prefill(K, V, None if imp is None else imp.cpu())
    for step in range(steps):
        kn, vn = make_token(w, step)
        q = make_q(w, step=step)
        a = fused.decode_step(kn.cuda(), vn.cuda(), q.cuda(), workspace=ws_f, importance=imp)
        split.append(kn.cuda(), vn.cuda())
        ref.append(kn, vn)
        if split.lengths()[1] == 128:
            split.flush(importance=imp)
            ref.flush(None if imp is None else imp.cpu())
        b = split.attention(q.cuda(), workspace=ws_s)
        assert fused.lengths() == split.lengths()
        assert fused.sink_tokens() == split.sink_tokens()
        assert torch.equal(a, b), f"step {step}: fused and separate outputs differ"
    for x, y in zip(fused.export_residual(), split.export_residual()):
        assert torch.equal(x, y)
    if mode == "uniform":
        for x, y in zip(fused.export_k() + fused.export_v(), split.export_k() + split.export_v()):
            assert torch.equal(x, y)
    assert_attention_close(a, ref.attention(q), f"decode step {w}")
    assert fused.status() == 0


def test_decode_step_rejects_a_full_residual_without_changes():
    """A residual already holding 128 tokens must be flushed first: the step
    returns RESIDUAL_FULL and leaves the lengths as they were."""
    w = Workload("step_full", 92, B=1, Hq=4, Hkv=1, T_q=0, r=128)
    K, V = make_kv(w, 128)
    cache = kvq.KVCache(1, 1, 512, 2, 2)
    cache.prefill(K[:, :, :127].contiguous().cuda(), V[:, :, :127].contiguous().cuda())
    kn, vn = make_token(w, 0)
    cache.append(kn.cuda(), vn.cuda())                 # r = 128
    with pytest.raises(kvq.KVQError) as e:
        cache.decode_step(kn.cuda(), vn.cuda(), make_q(w).cuda())
    assert e.value.name == "RESIDUAL_FULL"
    assert cache.lengths() == (0, 128)


def test_decode_split_event_brackets_the_decode_kernel_once():
    """kvq_set_decode_split_event: the next call records the event between
    its decode kernel and its combine (inside the call's own events), the
    output is the same as without it, and the call after forgets it."""
    w = Workload("split_event", 93, B=2, Hq=8, Hkv=2, T_q=0, r=1000, k_outliers=4)
    K, V = make_kv(w, 1000)
    cache = kvq.KVCache(2, 2, 1280)
    cache.prefill(K.cuda(), V.cuda())
    q = make_q(w).cuda()
    ws = cache.workspace(w.Hq)
    want = cache.attention(q, workspace=ws).clone()
    e0, mid, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record()
    kvq.set_decode_split_event(mid)
    got = cache.attention(q, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    t_mid, t_end = e0.elapsed_time(mid), e0.elapsed_time(e1)
    assert 0.0 < t_mid <= t_end
    # one-shot: the next call does not record it again
    cache.attention(q, workspace=ws)
    torch.cuda.synchronize()
    assert e0.elapsed_time(mid) == t_mid
    # a pending event can be cancelled
    kvq.set_decode_split_event(mid)
    kvq.set_decode_split_event(None)
    cache.attention(q, workspace=ws)
    torch.cuda.synchronize()
    assert e0.elapsed_time(mid) == t_mid
