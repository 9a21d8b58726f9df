"""Host logic of bench.py on the CPU: workload selection (sweep points by
name, overrides) and the algorithmic byte counts the roofline divides by."""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bit_kv_cache_kvq_gb300.workloads import WORKLOADS, sweep_workload  # noqa: E402


def _args(**kw):
    base = dict(workload="llama8b_gqa_32k_b16", batch=0, context=0, bits=0)
    base.update(kw)
    return argparse.Namespace(**base)


def test_sweep_points_by_name():
    for c, b, k in [(4096, 1, 2), (131072, 64, 4), (16384, 8, 2)]:
        w = bench.workload_from(_args(workload=f"sweep_c{c}_b{b}_k{k}"))
        ref = sweep_workload(c, b, k)
        assert (w.T_q, w.B, w.k_bits, w.v_bits, w.Hq, w.Hkv, w.r) == \
               (ref.T_q, ref.B, ref.k_bits, ref.v_bits, 32, 8, 100)


def test_overrides_apply_to_the_named_workload():
    w = bench.workload_from(_args(batch=8, context=4096, bits=4))
    assert (w.B, w.T_q, w.k_bits, w.v_bits) == (8, 4096, 4, 4)
    assert w.Hq == WORKLOADS["llama8b_gqa_32k_b16"].Hq


def test_algorithmic_bytes_per_token_and_call():
    """94 B per quantized token and KV head at 2 bits (K codes 32 + a bf16
    origin and fp32 step per channel over 128 tokens = 6; V codes 32 + an
    origin and step per 32-channel group = 24), 158 B at 4 bits, 512 B per
    residual token, q (bf16) and o (fp32) per query head: the Llama-8B
    GQA 32K x 16 call reads 401 211 392 B."""
    w = WORKLOADS["llama8b_gqa_32k_b16"]
    assert bench.token_bytes(w) == 94
    assert bench.token_bytes(sweep_workload(4096, 1, 4)) == 158
    assert bench.attention_bytes(w, 32768, 100) == 401_211_392
    mix = WORKLOADS["mixkvq_qwen32b_16k_b8"]
    assert bench.mixed_k_group_bytes(mix) == 7100
    assert bench.attention_bytes(mix, 16384, 100) == 120_553_472
