"""GPU parity: libkvq (through the C ABI) against the CPU oracle on the same
seeded inputs.  Codes, origins, steps bit-exact; attention within the
tolerance stated in kvq_testing."""
import numpy as np
import pytest
import torch

import oracle as orc
import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300 import _build
from bit_kv_cache_kvq_gb300.workloads import (WORKLOADS, Workload, bf16_bits, make_kv, make_q,
                                              make_token, scaled, sweep_workload)
from kvq_testing import UnitOracles, assert_attention_close, assert_uniform_exports_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    kvq.lib()


def small(B, Hkv, n_rep, T_q, r, k_bits=2, v_bits=2, seed=77) -> Workload:
    return Workload("small", seed, B=B, Hq=Hkv * n_rep, Hkv=Hkv, T_q=T_q, r=r,
                    k_bits=k_bits, v_bits=v_bits)


def run_case(w: Workload, extra_tokens: int = 0, device="cuda", gen_device="cpu",
             units=None, max_tokens=None, flush_when_full=True):
    """Prefill T - extra_tokens tokens, append extra_tokens (flushing when
    the residual is full, MixKVQ Algorithm 1 order), return (gpu cache,
    oracle caches, q)."""
    L = w.T - extra_tokens
    K, V = make_kv(w, L, device=gen_device)
    units = list(range(w.B * w.Hkv)) if units is None else units
    cap = max_tokens or (w.T_q + 128 * (1 + extra_tokens // 128))
    cache = kvq.KVCache(w.B, w.Hkv, cap, w.k_bits, w.v_bits)
    cache.prefill(K.to(device), V.to(device))
    ref = UnitOracles(units, w.Hkv, w.k_bits, w.v_bits)
    ref.prefill(K, V)
    for step in range(extra_tokens):
        kn, vn = make_token(w, step, device=gen_device)
        cache.append(kn.to(device), vn.to(device))
        ref.append(kn, vn)
        if flush_when_full and cache.lengths()[1] == 128:
            cache.flush()
            ref.flush()
    q = make_q(w, device=gen_device)
    return cache, ref, q


# ------------------------------------------------------------ quantization
@pytest.mark.parametrize("B,Hkv,L,kb,vb", [
    (1, 1, 128, 2, 2),
    (2, 2, 3 * 128 + 37, 2, 2),
    (2, 3, 2 * 128 + 127, 4, 4),
    (1, 2, 5 * 128, 2, 4),
    (2, 1, 100, 4, 2),          # shorter than one group: residual only
])
def test_prefill_codes_bit_exact(B, Hkv, L, kb, vb):
    w = small(B, Hkv, 1, L - L % 128, L % 128, kb, vb)
    cache, ref, _ = run_case(w)
    assert cache.lengths() == (L - L % 128, L % 128)
    assert_uniform_exports_equal(cache, ref)
    assert cache.status() == 0


@pytest.mark.parametrize("n_groups", [29, 30, 31, 61, 62])
def test_combine_row_sizes(n_groups):
    """Rows of 31, 32, 33, 63 and 64 partials (few units, so one split
    position per warp: a unit's groups, then its residual window weighted as
    two), on both sides of the combine kernels' limit (one round trip for up
    to 32 partials a row, 8 warps a row above)."""
    w = small(1, 2, 4, 128 * n_groups, 50)
    cache, ref, q = run_case(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), f"{n_groups} groups")


@pytest.mark.parametrize("B,Hkv,n_rep,n_groups", [
    (1, 2, 4, 150),     # 8 rows of ~300 partials: 16 warps a row
    (3, 8, 4, 200),     # 96 rows of ~100 partials: 6 warps a row
    (5, 8, 4, 80),      # 160 rows of ~60 partials: 4 warps a row
    (1, 1, 4, 700),     # 4 rows of 702 partials: up to three chunks a warp
    (1, 1, 4, 3000),    # one split position per resident warp: 2432 partials a row
])
def test_combine_many_partials(B, Hkv, n_rep, n_groups):
    """Rows of more than 32 partials (the many-partials combine) at row
    counts below, around and above the SM count."""
    w = small(B, Hkv, n_rep, 128 * n_groups, 77)
    cache, ref, q = run_case(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), f"{B * w.Hq} rows")


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4)])
def test_append_and_flush_bit_exact(kb, vb):
    # prefill 2 groups + 120 residual, then 8 appends fill the residual, one
    # flush seals it, and 3 more appends start the next window
    w = small(2, 2, 2, 3 * 128, 3, kb, vb)
    cache, ref, q = run_case(w, extra_tokens=11)
    assert cache.lengths() == (3 * 128, 3)
    assert_uniform_exports_equal(cache, ref)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "after flush")


def test_constant_and_special_groups():
    """Constant channels/tokens (step 0), -0.0 and +0.0 mixes, exact ties, and
    a record whose value groups are all constant (every value step 0)."""
    w = small(1, 2, 1, 256, 0)
    K, V = make_kv(w)
    K[0, 0, :128, 5] = 3.0                      # constant key channel
    K[0, 1, 128:, 7] = 0.0
    K[0, 1, 130, 7] = -0.0                      # signed zeros only
    V[0, 0, 10, :32] = -2.5                     # constant value group
    V[0, 1, 11, 32:64] = torch.tensor([0.0, 0.5, 2.5, 3.0] * 8)   # RNE ties
    V[0, 0, 128:, :] = 0.75                     # a whole record of constant value groups
    cache = kvq.KVCache(1, 2, 256, 2, 2)
    cache.prefill(K.cuda(), V.cuda())
    ref = UnitOracles([0, 1], 2)
    ref.prefill(K, V)
    assert_uniform_exports_equal(cache, ref)
    q = make_q(w)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "special groups")


# ---------------------------------------------------------------- decode
DECODE_CASES = [
    # (B, Hkv, n_rep, T_q, r, kb, vb)
    (1, 1, 1, 0, 1, 2, 2),
    (2, 2, 1, 128, 0, 2, 2),
    (2, 2, 2, 640, 37, 2, 2),
    (1, 2, 4, 1152, 127, 2, 2),
    (2, 1, 8, 256, 128, 2, 2),
    (1, 1, 4, 0, 128, 2, 2),
    (2, 2, 4, 640, 64, 4, 4),
    (1, 2, 8, 512, 5, 4, 4),
    (2, 2, 4, 384, 100, 2, 4),
    (1, 3, 2, 896, 1, 4, 2),
]


@pytest.mark.parametrize("B,Hkv,n_rep,T_q,r,kb,vb", DECODE_CASES)
def test_decode_attention_parity(B, Hkv, n_rep, T_q, r, kb, vb):
    w = small(B, Hkv, n_rep, T_q, r, kb, vb)
    extra = 1 if r == 128 else 0           # r = 128 is only reachable by appending
    cache, ref, q = run_case(w, extra_tokens=extra, flush_when_full=False)
    assert cache.lengths() == (T_q, r)
    out = cache.attention(q.cuda())
    assert_attention_close(out, ref.attention(q), f"decode {w}")


def test_decode_with_an_empty_split():
    """160 units x 5 groups: the split policy leaves the last split of each
    unit without groups; its partial must drop out of the merge."""
    w = small(20, 8, 1, 640, 0, seed=5)
    cache, ref, q = run_case(w, units=[0, 77, 159])
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), "empty split")


def test_decode_repeatable_and_workspace_reuse():
    w = small(2, 2, 4, 640, 37)
    cache, ref, q = run_case(w)
    ws = cache.workspace(w.Hq)
    a = cache.attention(q.cuda(), workspace=ws).clone()
    b = cache.attention(q.cuda(), workspace=ws)
    assert torch.equal(a, b)


@pytest.mark.parametrize("B,Hkv,n_rep,T_q,r", [
    (4, 8, 4, 1024, 50),    # 32 units of 9 items: a few partials a unit
    (1, 1, 4, 8192, 3),     # one unit of 65 items: 65 partials to merge
])
def test_decode_merge_of_partials(B, Hkv, n_rep, T_q, r):
    w = small(B, Hkv, n_rep, T_q, r, seed=41)
    units = None if B * Hkv <= 4 else [0, 13, 31]
    cache, ref, q = run_case(w, units=units)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), f"merge {w}")


def test_decode_workspace_needs_no_initial_contents():
    """Any prior workspace contents (here all bytes 0xff, then 0x00) give
    the same result: every partial the merge reads is written by the call."""
    w = small(4, 8, 4, 1024, 50, seed=42)
    cache, ref, q = run_case(w, units=[0, 31])
    want = ref.attention(q)
    for fill in (0xFF, 0x00, 0xFF):
        ws = cache.workspace(w.Hq)
        ws.fill_(fill)
        assert_attention_close(cache.attention(q.cuda(), workspace=ws), want, f"fill {fill:#x}")


def test_decode_replayed_as_a_cuda_graph():
    """A captured decode (decode kernel and its programmatic-dependent
    combine) replays correctly with new queries in the captured buffer."""
    w = small(4, 8, 4, 1024, 50, seed=43)
    cache, ref, _ = run_case(w, units=[0, 5, 31])
    qs = [make_q(w, step=i) for i in range(3)]
    q_dev = qs[0].cuda()
    out = torch.empty(w.B, w.Hq, 128, dtype=torch.float32, device="cuda")
    ws = cache.workspace(w.Hq)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cache.attention(q_dev, out=out, workspace=ws)   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cache.attention(q_dev, out=out, workspace=ws)
    for i in (1, 2, 0, 1):
        q_dev.copy_(qs[i].cuda())
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_attention_close(out, ref.attention(qs[i]), f"replay q{i}")


# ----------------------------------------------------- the named workloads
def test_tiny_single_head_workload():
    w = WORKLOADS["tiny_1head_1k"]
    cache, ref, q = run_case(w)
    assert cache.lengths() == (1024, 64)
    assert_uniform_exports_equal(cache, ref)
    assert_attention_close(cache.attention(q.cuda()), ref.attention(q), w.name)


def test_llama8b_32k_workload_sampled_units():
    """Full-size Llama-8B GQA decode layer (batch 16, 32768 + 100), in the
    launch configuration the benchmark times; the oracle checks three units."""
    w = WORKLOADS["llama8b_gqa_32k_b16"]
    units = [0, 61, 127]
    K, V = make_kv(w, device="cuda")
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128 * 64, w.k_bits, w.v_bits)
    cache.prefill(K, V)
    ref = UnitOracles(units, w.Hkv)
    ref.prefill(K, V)
    del K, V
    q = make_q(w, device="cuda")
    out = cache.attention(q)
    assert_uniform_exports_equal(cache, ref)
    assert_attention_close(out, ref.attention(q), w.name)
    assert cache.status() == 0


def test_prefill_flush_workload_sampled_units():
    """Prefill 32K at batch 8 (2-bit and 4-bit), then decode steps that cross
    a flush; checked on sampled units after the flush."""
    base = WORKLOADS["llama8b_prefill_32k_b8"]
    for bits in (2, 4):
        w = scaled(base, k_bits=bits, v_bits=bits)
        units = [3, 60]
        K, V = make_kv(w, device="cuda")
        cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128 * 5, bits, bits)
        cache.prefill(K, V)
        ref = UnitOracles(units, w.Hkv, bits, bits)
        ref.prefill(K, V)
        del K, V
        for step in range(130):
            kn, vn = make_token(w, step, device="cuda")
            cache.append(kn, vn)
            ref.append(kn, vn)
            if cache.lengths()[1] == 128:
                cache.flush()
                ref.flush()
        assert cache.lengths() == (w.T_q + 128, 2)
        assert_uniform_exports_equal(cache, ref)
        q = make_q(w, step=7, device="cuda")
        assert_attention_close(cache.attention(q), ref.attention(q), f"prefill {bits}-bit")


@pytest.mark.parametrize("context,batch,bits", [(4096, 1, 2), (4096, 8, 4), (131072, 8, 2),
                                                (65536, 1, 2), (131072, 64, 4)])
def test_sweep_points_sampled_units(context, batch, bits):
    """Long-context sweep points.  Small batches split over the whole GPU
    give each query row many partials (33 at 4K x 1; about 300 at 64K x 1,
    more than one pass of the 8-warp combine's 256-part stride); 128K x 64
    at 4 bits is the largest point (a 10.6 GB cache)."""
    w = sweep_workload(context, batch, bits)
    units = [0, w.B * w.Hkv - 1]
    K, V = make_kv(w, device="cuda")
    cache = kvq.KVCache(w.B, w.Hkv, w.T_q + 128, bits, bits)
    cache.prefill(K, V)
    ref = UnitOracles(units, w.Hkv, bits, bits)
    ref.prefill(K, V)
    del K, V
    q = make_q(w, device="cuda")
    assert_attention_close(cache.attention(q), ref.attention(q), w.name)


# --------------------------------------------------------- bf16 comparator
@pytest.mark.parametrize("T,n_rep", [(1, 1), (100, 4), (128, 8), (300, 4), (4096 + 17, 2)])
def test_bf16_decode_parity(T, n_rep):
    w = small(2, 2, n_rep, T, 0)
    K, V = make_kv(w, T)
    q = make_q(w)
    out = kvq.decode_bf16(K.cuda(), V.cuda(), q.cuda())
    ref = np.zeros((w.B, w.Hq, 128))
    kf = orc.bf16_to_f32(bf16_bits(K)).astype(np.float64)
    vf = orc.bf16_to_f32(bf16_bits(V)).astype(np.float64)
    qf = orc.bf16_to_f32(bf16_bits(q)).astype(np.float64)
    for b in range(w.B):
        for h in range(w.Hq):
            ref[b, h] = orc.attention(qf[b, h], kf[b, h // n_rep], vf[b, h // n_rep])
    assert_attention_close(out, ref, "bf16")


# ----------------------------------------------------------------- saliency
@pytest.mark.parametrize("B,Hkv,n_rep,Lq", [(2, 2, 8, 128), (1, 3, 4, 17), (2, 1, 1, 1)])
def test_saliency_bit_exact(B, Hkv, n_rep, Lq):
    w = scaled(WORKLOADS["mixkvq_qwen32b_16k_b8"], B=B, Hkv=Hkv, Hq=Hkv * n_rep, Lq=Lq, T_q=128, r=0)
    from bit_kv_cache_kvq_gb300.workloads import make_query_window
    qw = make_query_window(w)
    K, _ = make_kv(w, 128)
    I, A, tiers = kvq.channel_saliency(qw.cuda(), K.cuda(), 2, n_bf16=6, n_uint4=25)
    I2, A2, tiers_t = kvq.channel_saliency(qw.cuda(), K.cuda(), 2, tau_bf16=1.5, tau_uint4=0.6)
    torch.cuda.synchronize()
    for b in range(B):
        for h in range(Hkv):
            Iref = orc.importance(bf16_bits(qw[b, h * n_rep:(h + 1) * n_rep]))
            Sref = orc.sensitivity(bf16_bits(K[b, h]), 2)
            Aref = orc.salience(Iref, Sref)
            assert np.array_equal(I[b, h].cpu().numpy().view(np.uint32), Iref.view(np.uint32))
            assert np.array_equal(A[b, h].cpu().numpy().view(np.uint32), Aref.view(np.uint32))
            assert np.array_equal(tiers[b, h].cpu().numpy(), orc.tiers_rank(Aref, 6, 25))
            assert np.array_equal(tiers_t[b, h].cpu().numpy(), orc.tiers_threshold(Aref, 1.5, 0.6))


# ------------------------------------------------------ errors and flags
def test_state_machine_errors():
    w = small(1, 1, 1, 0, 0)
    cache = kvq.KVCache(1, 1, 256)
    q = make_q(w).cuda()
    with pytest.raises(kvq.KVQError) as e:
        cache.attention(q)
    assert e.value.name == "EMPTY"
    with pytest.raises(kvq.KVQError) as e:
        cache.flush()
    assert e.value.name == "RESIDUAL_NOT_FULL"
    K, V = make_kv(small(1, 1, 1, 256, 0))
    cache.prefill(K.cuda(), V.cuda())
    with pytest.raises(kvq.KVQError) as e:
        cache.prefill(K.cuda(), V.cuda())
    assert e.value.name == "NOT_EMPTY"
    kn, vn = make_token(w, 0)
    for _ in range(128):
        cache.append(kn.cuda(), vn.cuda())
    with pytest.raises(kvq.KVQError) as e:
        cache.append(kn.cuda(), vn.cuda())
    assert e.value.name == "RESIDUAL_FULL"
    with pytest.raises(kvq.KVQError) as e:
        cache.flush()                        # 256 + 128 > capacity 256
    assert e.value.name == "CAPACITY"
    assert cache.lengths() == (256, 128)     # unchanged by the failed calls
    with pytest.raises(kvq.KVQError) as e:
        cache.attention(make_q(small(1, 1, 3, 0, 0)).cuda())   # 3 heads per KV head
    assert e.value.name == "SHAPE"
    small_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        cache.attention(q, workspace=small_ws)
    assert e.value.name == "WORKSPACE"


def test_nonfinite_and_range_flags():
    w = small(1, 1, 1, 128, 0)
    K, V = make_kv(w)
    K[0, 0, 5, 9] = float("nan")
    cache = kvq.KVCache(1, 1, 128)
    cache.prefill(K.cuda(), V.cuda())
    assert cache.status() & kvq.FLAG_NONFINITE
    K, V = make_kv(w)
    V[0, 0, 3, 0] = 3.0e38
    V[0, 0, 3, 1] = -3.0e38                  # range overflows fp32
    cache2 = kvq.KVCache(1, 1, 128)
    cache2.prefill(K.cuda(), V.cuda())
    assert cache2.status() == kvq.FLAG_RANGE
    with pytest.raises(orc.OracleError):     # the oracle rejects the same group
        orc.quantize_group(orc.bf16_to_f32(bf16_bits(V[0, 0, 3, :32])), 2)
