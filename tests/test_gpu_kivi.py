"""KIVI streaming variant on the GPU ("KIVI: KV cache axes" §4–§7): keys in
32-token groups sealed every 128 tokens, values a 128-token FIFO whose
oldest token leaves quantized per token over 32 channels, bf16 metadata
computed in bf16.  The cache state is compared bit for bit with the
oracle's KiviOracleCache (key codes, origins and steps per 32-token group;
value codes, origins and steps per token; the key residual; the FIFO
oldest first) after a prefill and across appends that seal keys and pop the
FIFO; the attention output within the stated tolerance of the oracle's fp64
attention over its own dequantized cache."""
import numpy as np
import pytest
import torch

import oracle as orc
import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import Workload, bf16_bits, make_kv, make_q, make_token
from kvq_testing import assert_attention_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


def assert_kivi_state_equal(cache: kvq.KVCache, ref: orc.KiviOracleCache, where: str):
    st = {k: v.cpu() for k, v in cache.export_kivi().items()}
    torch.cuda.synchronize()
    bits = cache.k_bits
    B, H = cache.batch, cache.kv_heads
    tk, rk = cache.lengths()
    for u in range(B * H):
        b, h = divmod(u, H)
        ntk, nrk, ntv, nrv = ref.lengths(u)
        assert (tk, rk) == (ntk, nrk), f"{where}: key lengths {tk, rk} vs {ntk, nrk}"
        kc = st["k_codes"][b, h].numpy()
        ko, ks = bf16_bits(st["k_origin"][b, h]), bf16_bits(st["k_step"][b, h])
        assert kc.shape[0] == len(ref.kq[u])
        for gi, (codes, origin, step) in enumerate(ref.kq[u]):
            want = np.stack([np.frombuffer(orc.pack_lsb(codes[:, d], bits), np.uint8)
                             for d in range(codes.shape[1])])
            assert np.array_equal(kc[gi], want), f"{where}: key codes differ (unit {u}, group {gi})"
            assert np.array_equal(ko[gi], origin), f"{where}: key origins differ (unit {u}, group {gi})"
            assert np.array_equal(ks[gi], step), f"{where}: key steps differ (unit {u}, group {gi})"
        vc = st["v_codes"][b, h].numpy()
        vo, vs = bf16_bits(st["v_origin"][b, h]), bf16_bits(st["v_step"][b, h])
        assert ntv == len(ref.vq[u]) and ntv <= vc.shape[0]
        for t, (codes, origin, step) in enumerate(ref.vq[u]):
            want = np.frombuffer(orc.pack_lsb(codes, bits), np.uint8)
            assert np.array_equal(vc[t], want), f"{where}: value codes differ (unit {u}, token {t})"
            assert np.array_equal(vo[t], origin), f"{where}: value origins differ (unit {u}, token {t})"
            assert np.array_equal(vs[t], step), f"{where}: value steps differ (unit {u}, token {t})"
        assert not vc[ntv:].any() and not vo[ntv:].any() and not vs[ntv:].any(), \
            f"{where}: rows of FIFO tokens not zero (unit {u})"
        kr = bf16_bits(st["k_res"][b, h])
        vr = bf16_bits(st["v_res"][b, h])
        assert np.array_equal(kr, np.asarray(ref.kr[u], np.uint16).reshape(-1, 128)), \
            f"{where}: key residual differs (unit {u})"
        assert np.array_equal(vr, np.asarray(ref.vr[u], np.uint16).reshape(-1, 128)), \
            f"{where}: value FIFO differs (unit {u})"


@pytest.mark.parametrize("B,Hkv,n_rep,L,steps,bits", [
    (1, 2, 4, 40, 100, 2),        # FIFO not yet full, first seal during the steps
    (2, 2, 4, 128, 140, 2),       # prefill seals one record; the FIFO pops every step
    (1, 3, 8, 300, 90, 4),        # 2 records + 44, 4-bit, 8 query heads per KV head
    (2, 1, 1, 1000, 150, 2),      # 7 records + 104, a seal after 24 steps
    (1, 2, 2, 257, 10, 4),
])
def test_kivi_state_and_attention_match_oracle(B, Hkv, n_rep, L, steps, bits):
    w = Workload("kivi", 1101, B=B, Hq=Hkv * n_rep, Hkv=Hkv, T_q=0, r=L, k_bits=bits,
                 v_bits=bits, k_outliers=4)
    K, V = make_kv(w, L)
    cap = 128 * ((L + steps) // 128 + 2)
    cache = kvq.KVCache(B, Hkv, cap, bits, bits, mode="kivi")
    cache.prefill(K.cuda(), V.cuda())
    ref = orc.KiviOracleCache(B, Hkv, 128, bits, bits)
    ref.prefill(bf16_bits(K), bf16_bits(V))
    assert_kivi_state_equal(cache, ref, "prefill")
    q = make_q(w, step=0)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(bf16_bits(q)), "prefill")
    ws = cache.workspace(w.Hq)
    checks = {steps - 1} | {s for s in range(steps) if (L + s + 1) % 128 in (0, 1, 77)}
    for step in range(steps):
        kn, vn = make_token(w, step)
        q = make_q(w, step=step + 1)
        out = cache.decode_step(kn.cuda(), vn.cuda(), q.cuda(), workspace=ws)
        ref.append(bf16_bits(kn), bf16_bits(vn))
        if step in checks:
            assert_kivi_state_equal(cache, ref, f"step {step}")
            assert_attention_close(out, ref.attention(bf16_bits(q)), f"step {step}")
    assert cache.status() == 0


def test_kivi_flush_is_a_mode_error_and_appends_seal():
    w = Workload("kivi_seal", 1102, B=1, Hq=4, Hkv=1, T_q=0, r=127, k_outliers=0)
    K, V = make_kv(w, 127)
    cache = kvq.KVCache(1, 1, 512, mode="kivi")
    cache.prefill(K.cuda(), V.cuda())
    assert cache.lengths() == (0, 127)
    with pytest.raises(kvq.KVQError) as e:
        cache.flush()
    assert e.value.name == "MODE"
    kn, vn = make_token(w, 0)
    cache.append(kn.cuda(), vn.cuda())
    assert cache.lengths() == (128, 0)          # the 128th key sealed the residual
    ref = orc.KiviOracleCache(1, 1, 128)
    ref.prefill(bf16_bits(K), bf16_bits(V))
    ref.append(bf16_bits(kn), bf16_bits(vn))
    assert_kivi_state_equal(cache, ref, "after the seal")
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(bf16_bits(q)), "after the seal")
