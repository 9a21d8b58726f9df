"""PN-Mix H3/L1 keys on the GPU (PN-Mix reproduction notes, Eq. 2, Eq. 6,
Eq. 7, App. G): the Eq. 6 pair scores and the selection of the 3-bit pairs,
then the key groups (3-bit codes for the selected pairs' channels, one bit
with the midpoint correction for the others; offsets and scales) compared
with the oracle bit for bit after a prefill and after flushes, the values
as in the uniform cache, and the attention within the stated tolerance of
the oracle's fp64 attention over its own dequantized cache."""
import numpy as np
import pytest
import torch

import oracle as orc
import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, bf16_bits, make_kv, make_q, make_token
from kvq_testing import assert_attention_close, f32_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


def query_window(B, Hq, Lq, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, 128, generator=g)
    q[..., 5] *= 6.0                      # a few large-|q| channels
    q[..., 70] *= 4.0
    return q.to(torch.bfloat16)


@pytest.mark.parametrize("B,Hkv,n_rep,L,steps,n_high,layout,vb", [
    (1, 2, 4, 256 + 40, 100, 32, 0, 2),     # r = 0.5, adjacent pairs; a flush during the steps
    (2, 1, 8, 384 + 3, 140, 32, 1, 2),      # split halves (Hugging Face layout), 8 heads
    (1, 2, 1, 128, 130, 16, 0, 4),          # 4-bit values, one flush
    (1, 1, 4, 256, 10, 0, 0, 2),            # no 3-bit pairs: all channels one bit
    (1, 1, 2, 256, 10, 64, 1, 2),           # every pair 3-bit
])
def test_pnmix_pairs_groups_and_attention(B, Hkv, n_rep, L, steps, n_high, layout, vb):
    w = Workload("pnmix", 1201, B=B, Hq=Hkv * n_rep, Hkv=Hkv, T_q=0, r=L, v_bits=vb,
                 k_outliers=4)
    K, V = make_kv(w, L)
    Lq = 64
    qwin = query_window(B, w.Hq, Lq, 1202)
    cache = kvq.KVCache(B, Hkv, 128 * ((L + steps) // 128 + 2), 2, vb, mode="pnmix",
                        n_high_pairs=n_high, pair_layout=layout)
    sigma = cache.pnmix_pairs(qwin.cuda(), K.cuda()).cpu().numpy()
    cache.prefill(K.cuda(), V.cuda())
    # Eq. 6 scores and the selection, bit for bit
    high = np.zeros((B, Hkv, 128), bool)
    for b in range(B):
        for h in range(Hkv):
            ref_sigma = orc.pair_scores(bf16_bits(qwin[b, h * n_rep:(h + 1) * n_rep]),
                                        bf16_bits(K[b, h]), layout)
            assert np.array_equal(sigma[b, h].view(np.uint32), ref_sigma.view(np.uint32)), \
                f"pair scores differ (unit {b, h})"
            high[b, h] = orc.channel_mask(orc.select_pairs(ref_sigma, n_high), layout)
    ref = orc.OracleCache(B, Hkv, 128, 2, vb, mode="pnmix", high_channels=high)
    ref.prefill(bf16_bits(K), bf16_bits(V))

    def check(where, q):
        codes, off, sc, hi = (t.cpu() for t in cache.export_pnmix())
        vc, vm, vs = cache.export_v()
        torch.cuda.synchronize()
        assert np.array_equal(hi.numpy().astype(bool), high), f"{where}: high channels differ"
        vc, vm, vs = vc.cpu().numpy(), bf16_bits(vm), f32_bits(vs)
        for u in range(B * Hkv):
            b, h = divmod(u, Hkv)
            assert codes.shape[2] == len(ref.k_groups[u])
            for gi, (c, o, s) in enumerate(ref.k_groups[u]):
                assert np.array_equal(codes[b, h, gi].numpy(), c), f"{where}: codes (unit {u}, group {gi})"
                assert np.array_equal(f32_bits(off[b, h, gi]), o.view(np.uint32)), \
                    f"{where}: offsets (unit {u}, group {gi})"
                assert np.array_equal(f32_bits(sc[b, h, gi]), s.view(np.uint32)), \
                    f"{where}: scales (unit {u}, group {gi})"
            if ref.v_parts[u]:
                ovc, ovm, ovs = (np.concatenate([p[i] for p in ref.v_parts[u]]) for i in range(3))
                assert np.array_equal(vc[b, h], ovc) and np.array_equal(vm[b, h], ovm) and \
                    np.array_equal(vs[b, h], ovs.view(np.uint32)), f"{where}: values (unit {u})"
        assert_attention_close(cache.attention(q.cuda()), ref.attention(bf16_bits(q)), where)

    check("prefill", make_q(w))
    ws = cache.workspace(w.Hq)
    for step in range(steps):
        kn, vn = make_token(w, step)
        q = make_q(w, step=step + 1)
        out = cache.decode_step(kn.cuda(), vn.cuda(), q.cuda(), workspace=ws)
        ref.append(bf16_bits(kn), bf16_bits(vn))
        if ref.r == 128:
            ref.flush()
            check(f"flush at step {step}", q)
            assert_attention_close(out, ref.attention(bf16_bits(q)), f"step {step}")
    assert_attention_close(out, ref.attention(bf16_bits(q)), "last step")
    assert cache.status() == 0


def test_pnmix_needs_pairs_before_prefill():
    cache = kvq.KVCache(1, 1, 512, 2, 2, mode="pnmix", n_high_pairs=32)
    K, V = make_kv(Workload("pn_order", 1203, B=1, Hq=1, Hkv=1, T_q=0, r=256), 256)
    with pytest.raises(kvq.KVQError) as e:
        cache.prefill(K.cuda(), V.cuda())
    assert e.value.name == "EMPTY"
