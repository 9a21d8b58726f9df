"""Pins for the CPU oracle: values the pages print, closed forms, invariants
and brute force — never the oracle's own formula retyped.

Each fixture under tests/golden/ carries its citation in its "source" field.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def frac(s):
    """Parse "a/b" or a number from a fixture."""
    if isinstance(s, str) and "/" in s:
        a, b = s.split("/")
        return Fraction(int(a), int(b))
    return Fraction(s)


def bf16_trunc(x):
    """bf16 bit patterns of x (float32 truncated to its top 16 bits)."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def qdq_rows(mat, bits):
    """Per-row groups (Value per-token axis) via the unit-level V quantizer."""
    m = np.asarray(mat, np.float32)
    T, D = m.shape
    codes, vmin, vscale = orc.quantize_v_unit(orc.f32_to_bf16_exact(m), D, bits)
    return orc.dequant_v_unit(codes, vmin, vscale, D, bits)


def qdq_cols(mat, bits):
    """Per-column groups (Key per-channel axis) via the unit-level K quantizer."""
    m = np.asarray(mat, np.float32)
    T, D = m.shape
    codes, kmin, kscale = orc.quantize_k_unit(orc.f32_to_bf16_exact(m), T, bits)
    return orc.dequant_k_unit(codes, kmin, kscale, T, bits)


# ------------------------------------------------------------ KIVI §3 Key
def test_key_example_per_token_row0():
    g = golden("kivi_key_4x4.json")
    row0 = g["key"][0]
    codes, m, s = orc.quantize_group(row0, g["bits"])
    assert list(codes) == [3, 0, 0, 0]
    assert m == -1.0
    # step is the fp32 rounding of 101/3 (fp32 step reading)
    assert s == np.float32(101.0) / np.float32(3.0)
    assert abs(Fraction(float(s)) - frac(g["per_token_row0_step"])) < Fraction(1, 2**19)
    rec = qdq_rows(g["key"], g["bits"])[0]
    np.testing.assert_allclose(rec, g["per_token_row0_reconstruction"], rtol=0, atol=1e-5)


def test_key_example_per_channel_reconstructs_exactly():
    g = golden("kivi_key_4x4.json")
    rec = qdq_cols(g["key"], g["bits"])
    assert np.array_equal(rec, np.asarray(g["key"], np.float64))
    for col, grid in zip(range(2), g["per_channel_column_grids"]):
        codes, m, s = orc.quantize_group([r[col] for r in g["key"]], 2)
        assert sorted(orc.dequantize_group(np.arange(4), m, s)) == grid


def _probs(keys, q):
    D = len(q)
    n = len(keys)
    _, p = orc.attention(q, np.asarray(keys, np.float64), np.zeros((n, D)), p_out=True)
    return p


def test_key_example_attention_decision():
    g = golden("kivi_key_4x4.json")
    q = g["query"]
    p_orig = _probs(g["key"], q)
    p_tok = _probs(qdq_rows(g["key"], 2), q)
    p_chan = _probs(qdq_cols(g["key"], 2), q)
    assert np.array_equal(p_chan, p_orig)
    assert int(np.argmax(p_orig)) == g["argmax_original"]
    assert int(np.argmax(p_tok)) == g["argmax_per_token"]
    assert np.max(np.abs(p_orig - p_tok)) > g["min_prob_change_per_token"]


# ---------------------------------------------------------- KIVI §3 Value
def test_value_example_axes():
    g = golden("kivi_value_4x4.json")
    p = np.asarray(g["p"])
    out_tok = p @ qdq_rows(g["value"], g["bits"])
    out_col = p @ qdq_cols(g["value"], g["bits"])
    # codes of the selected row are exact; with an fp32 step the top grid
    # point m + 3*fl32(1/3) differs from 1 by the step's rounding only
    codes, m, s = orc.quantize_group(g["value"][1], g["bits"])
    assert list(codes) == [3, 0, 3, 0] and m == 0.0
    np.testing.assert_allclose(out_tok, g["per_token_output"], rtol=0, atol=3 * 2.0**-24)
    target = float(frac(g["per_column_output_each"]))
    # fp32 step 200/3 carries a relative error below 2^-24
    np.testing.assert_allclose(out_col, [target] * 4, rtol=1e-6)
    codes, m, s = orc.quantize_group([r[1] for r in g["value"]], 2)
    assert abs(Fraction(float(s)) - frac(g["per_column_step"])) < Fraction(1, 2**16)


# --------------------------------------------------------------- KIVI §2
def test_two_bit_grid_has_no_zero():
    g = golden("kivi_grid_2bit.json")
    lo, hi = g["range"]
    codes, m, s = orc.quantize_group([lo, hi], g["bits"])
    grid = orc.dequantize_group(np.arange(4), m, s)
    for got, want in zip(grid, g["grid"]):
        assert abs(got - float(frac(want))) < 1e-7
    assert not np.any(grid == 0.0)


def test_constant_groups_exact():
    g = golden("kivi_constant_groups.json")
    for grp in g["groups"]:
        codes, m, s = orc.quantize_group(grp, g["bits"])
        assert list(orc.dequantize_group(codes, m, s)) == grp
        assert list(codes) == [0] * len(grp) and s == 0.0


def test_pack2_layout():
    g = golden("kivi_pack2.json")
    codes, _, _ = orc.quantize_group([100.0, 101.0, 102.0, 103.0], 2)
    assert list(codes) == g["codes_first_column"]
    packed = orc.pack_lsb(codes, 2)
    assert packed.hex() == g["packed_first_column_hex"]
    assert list(orc.unpack_lsb(packed, 4, 2)) == g["codes_first_column"]
    short = orc.pack_lsb(g["short_codes"], 2)
    assert len(short) == 1
    assert list(orc.unpack_lsb(short, g["short_length"], 2)) == g["short_codes"]
    with pytest.raises(ValueError):
        orc.unpack_lsb(short, 5, 2)


def test_four_bit_packing_low_nibble_first():
    # 4-bit analogue of the LSB-first rule: two codes per byte, first code low.
    assert orc.pack_lsb([0x3, 0xA, 0xF], 4).hex() == "a30f"


def test_round_half_to_even():
    # step 1 exactly: (x - m)/step lands on the ties 0.5 and 2.5
    codes, m, s = orc.quantize_group([0.0, 0.5, 2.5, 3.0], 2)
    assert s == 1.0
    assert list(codes) == [0, 0, 2, 3]     # half-away-from-zero gives [0,1,3,3]


def test_rejects_nonfinite_and_unrepresentable_step():
    with pytest.raises(orc.OracleError) as e:
        orc.quantize_group([0.0, float("nan"), 1.0], 2)
    assert e.value.status == orc.ORC_ERR_NONFINITE
    with pytest.raises(orc.OracleError) as e:
        orc.quantize_group([0.0, float("inf")], 2)
    assert e.value.status == orc.ORC_ERR_NONFINITE
    big = float(np.finfo(np.float32).max)
    with pytest.raises(orc.OracleError) as e:
        orc.quantize_group([-big, big], 2)
    assert e.value.status == orc.ORC_ERR_RANGE


# ---------------------------------------- MixKVQ appendix: error bound, brute force
@pytest.mark.parametrize("bits", [2, 4])
def test_error_bound_half_step(bits):
    g = golden("mixkvq_error_bound.json")
    rng = np.random.default_rng(7 + bits)
    for n in (4, 32, 128):
        for trial in range(50):
            x = (rng.standard_normal(n) * rng.choice([1e-3, 1.0, 30.0])).astype(np.float32)
            if trial % 7 == 0:
                x[rng.integers(n)] *= 40.0                       # an outlier
            codes, m, s = orc.quantize_group(x, bits)
            rec = orc.dequantize_group(codes, m, s)
            # fp32 (x - m) and division each round once: <= (2^b-1)*2^-23 steps
            slack = (2**bits - 1) * 2.0**-22
            assert np.all(np.abs(x.astype(np.float64) - rec) <= float(s) * (g["bound_fraction_of_step"] + slack))


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codes_brute_force_nearest(bits):
    """Every code is a nearest grid point of the exact (x - m)/step; exact
    ties (representable without rounding) go to the even code.  Three bits
    are PN-Mix's high channels (Eq. 2)."""
    rng = np.random.default_rng(100 + bits)
    top = 2**bits - 1
    for trial in range(300):
        n = int(rng.integers(2, 9))
        x = (rng.integers(-40, 40, n) / rng.choice([1, 2, 4, 8])).astype(np.float32)
        if trial % 3 == 0:
            x = rng.standard_normal(n).astype(np.float32)
        if x.max() == x.min():
            continue
        codes, m, s = orc.quantize_group(x, bits)
        for xi, c in zip(x, codes):
            y = (Fraction(float(xi)) - Fraction(float(m))) / Fraction(float(s))
            dists = [abs(y - k) for k in range(top + 1)]
            best = min(dists)
            assert dists[int(c)] <= best + Fraction(1, 2**20)
            if best == Fraction(1, 2) and dists[int(c)] == best and y.denominator == 2:
                assert int(c) % 2 == 0


# ---------------------------------------------------------- attention pins
def test_global_softmax_example():
    g = golden("kivi_global_softmax.json")
    q = [math.sqrt(2.0), 0.0]
    K = np.array([[0.0, 0.0]] * g["key_quant_rows"] + [[math.log(9.0), 0.0]])
    V = np.array([[float(t), -float(t)] for t in g["value_rows_first_dim"]])
    o, p = orc.attention(q, K, V, p_out=True)
    for got, want in zip(p, g["probabilities"]):
        assert abs(got - float(frac(want))) < 1e-12
    assert abs(o[0] - float(frac(g["output_first_dim"]))) < 1e-12
    assert abs(o[0] - g["output_first_dim_decimal"]) < 1e-6
    vb = g["value_boundary"]
    mixed = p[:vb] @ V[:vb] + p[vb:] @ V[vb:]
    assert np.allclose(mixed, o, atol=1e-12, rtol=0)
    kb = g["key_boundary"]
    # normalising the two Key segments separately is the page's wrong answer
    wrong = orc.attention(q, K[:kb], V[:kb])[0] + orc.attention(q, K[kb:], V[kb:])[0]
    assert abs(wrong - g["separate_softmax_output_first_dim"]) < 1e-12
    assert abs(wrong - o[0]) > 1.0


def test_attention_brute_force_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(3)
    for trial in range(40):
        n = int(rng.integers(1, 9))
        D = int(rng.choice([1, 2, 3, 4, 8]))
        q = rng.standard_normal(D) * 2
        K = rng.standard_normal((n, D)) * 3
        V = rng.standard_normal((n, D))
        o = orc.attention(q, K, V)
        # softmax without a max shift, 40 significant digits
        e = [mpmath.e ** (mpmath.fsum(mpmath.mpf(q[d]) * mpmath.mpf(K[t, d]) for d in range(D))
                          / mpmath.sqrt(D)) for t in range(n)]
        tot = mpmath.fsum(e)
        for d in range(D):
            ref = mpmath.fsum(e[t] * mpmath.mpf(V[t, d]) for t in range(n)) / tot
            assert abs(o[d] - float(ref)) <= 1e-13 * (1 + abs(float(ref)))


def test_output_error_decomposition_identity():
    """KIVI §1: o^ - o = (p^ - p) V + p^ E_V, with K^ = K + E_K, V^ = V + E_V."""
    rng = np.random.default_rng(11)
    n, D = 37, 16
    q = rng.standard_normal(D)
    K = rng.standard_normal((n, D))
    V = rng.standard_normal((n, D))
    EK = rng.standard_normal((n, D)) * 0.05
    EV = rng.standard_normal((n, D)) * 0.05
    o, p = orc.attention(q, K, V, p_out=True)
    oh, ph = orc.attention(q, K + EK, V + EV, p_out=True)
    assert np.allclose(oh - o, (ph - p) @ V + ph @ EV, atol=1e-12, rtol=0)


def test_attention_special_cases():
    rng = np.random.default_rng(5)
    D = 8
    v = rng.standard_normal((1, D))
    assert np.allclose(orc.attention(rng.standard_normal(D), rng.standard_normal((1, D)), v), v[0])
    V = rng.standard_normal((6, D))
    assert np.allclose(orc.attention(np.zeros(D), rng.standard_normal((6, D)), V), V.mean(0))
    # shift invariance: adding a constant logit to every row changes nothing
    q = np.zeros(D); q[0] = 1.0
    K = rng.standard_normal((6, D))
    K2 = K.copy(); K2[:, 0] += 5.0
    assert np.allclose(orc.attention(q, K, V), orc.attention(q, K2, V), atol=1e-12)


# ------------------------------------------------------------ state machine
def test_residual_trace_block_flush():
    g = golden("kivi_residual_trace.json")
    R, G, D = g["R"], g["G"], 4
    cache = orc.OracleCache(1, 1, D, Gk=G, Gv=D, R=R)
    rng = np.random.default_rng(0)
    lengths = []
    for step in range(g["steps"]):
        kv = orc.f32_to_bf16_exact(rng.integers(-8, 8, (2, 1, 1, D)).astype(np.float32))
        cache.append(kv[0], kv[1])
        if cache.r == R:
            cache.flush()
        lengths.append(cache.r)
    assert lengths == g["persisted_key_residual_lengths"]
    assert [cache.T_q, cache.r] == g["step9_key_split"]
    with pytest.raises(ValueError):
        cache.flush()                          # residual not full


def test_state_machine_errors_and_prefill_split():
    D = 8
    cache = orc.OracleCache(1, 1, D, Gk=4, Gv=8, R=4)
    rng = np.random.default_rng(1)
    KV = orc.f32_to_bf16_exact(rng.integers(-8, 8, (2, 1, 1, 10, D)).astype(np.float32))
    with pytest.raises(ValueError):
        cache.attention(KV[0][:, :, 0])        # empty cache
    cache.prefill(KV[0], KV[1])
    assert (cache.T_q, cache.r) == (8, 2)      # r = 10 mod 4
    with pytest.raises(ValueError):
        cache.prefill(KV[0], KV[1])            # not empty
    for _ in range(2):
        cache.append(KV[0][:, :, 0], KV[1][:, :, 0])
    with pytest.raises(ValueError):
        cache.append(KV[0][:, :, 0], KV[1][:, :, 0])   # full: flush first


def test_cache_attention_reduces_to_textbook_without_history():
    """T_q = 0: attention over the bf16 residual alone is textbook softmax."""
    rng = np.random.default_rng(2)
    D, r, Hq = 16, 5, 2
    cache = orc.OracleCache(1, 1, D, Gk=8, Gv=8, R=8)
    K = orc.f32_to_bf16_exact(rng.integers(-6, 6, (1, 1, r, D)).astype(np.float32))
    V = orc.f32_to_bf16_exact(rng.integers(-6, 6, (1, 1, r, D)).astype(np.float32))
    cache.prefill(K, V)
    q = orc.f32_to_bf16_exact(rng.integers(-3, 3, (1, Hq, D)).astype(np.float32))
    out = cache.attention(q)
    kf = orc.bf16_to_f32(K[0, 0]).astype(np.float64)
    vf = orc.bf16_to_f32(V[0, 0]).astype(np.float64)
    for h in range(Hq):
        s = kf @ orc.bf16_to_f32(q[0, h]).astype(np.float64) / np.sqrt(D)
        w = np.exp(s - s.max()); w /= w.sum()
        assert np.allclose(out[0, h], w @ vf, atol=1e-12)


def test_canonical_k_layout_channel_codes_along_tokens():
    """K codes: group g, channel d holds that channel's G codes packed LSB
    first along tokens (PN-Mix App. G; KIVI §3 packer)."""
    T, D, G = 8, 3, 4
    k = np.zeros((T, D), np.float32)
    k[:, 1] = [0, 1, 2, 3, 3, 2, 1, 0]           # channel 1: codes are the values
    k[:, 0] = 7.0                                # constant channel
    k[:, 2] = [0, 3, 0, 3, 1, 1, 1, 4]
    codes, kmin, kscale = orc.quantize_k_unit(orc.f32_to_bf16_exact(k), G, 2)
    assert codes.shape == (2, 3, 1)
    assert codes[0, 1, 0] == 0b11100100 and codes[1, 1, 0] == 0b00011011
    assert codes[0, 0, 0] == 0 and kscale[0, 0] == 0.0 and orc.bf16_to_f32(kmin[0, 0]) == 7.0
    assert list(orc.unpack_lsb(bytes(codes[0, 2]), 4, 2)) == [0, 3, 0, 3]


# ---------------------------------------------------------------- saliency
def test_saliency_hand_computed():
    """MixKVQ: I_d = mean |Q_{i,d}| over the GQA group's heads and the window,
    S_d = (max - min)/(2^B - 1), A_d = I_d * S_d — on integer inputs whose
    results are exact."""
    n_rep, Lq, D = 2, 2, 4
    Q = np.zeros((n_rep, Lq, D), np.float32)
    Q[:, :, 0] = [[1, -2], [3, -4]]      # sum |.| 10 -> I 2.5
    Q[:, :, 1] = [[0, 0], [0, 8]]        # 8 -> 2
    Q[:, :, 2] = [[-1, -1], [-1, -1]]    # 4 -> 1
    Q[:, :, 3] = [[2, 2], [2, 2]]        # 8 -> 2
    I = orc.importance(orc.f32_to_bf16_exact(Q))
    assert list(I) == [2.5, 2.0, 1.0, 2.0]
    K = np.zeros((4, D), np.float32)
    K[:, 0] = [0, 3, 1, 2]               # range 3 -> S 1
    K[:, 1] = [-6, 0, 0, 0]              # range 6 -> S 2
    K[:, 2] = [5, 5, 5, 5]               # range 0 -> S 0
    K[:, 3] = [1, 2, 3, 4]               # range 3 -> S 1
    S = orc.sensitivity(orc.f32_to_bf16_exact(K), 2)
    assert list(S) == [1.0, 2.0, 0.0, 1.0]
    A = orc.salience(I, S)
    assert list(A) == [2.5, 4.0, 0.0, 2.0]
    # rank form: one BF16, one UINT4, the rest UINT2
    assert list(orc.tiers_rank(A, 1, 1)) == [orc.TIER_UINT4, orc.TIER_BF16,
                                             orc.TIER_UINT2, orc.TIER_UINT2]
    # threshold form: strict ">" at both thresholds
    assert list(orc.tiers_threshold(A, 2.5, 2.0)) == [orc.TIER_UINT4, orc.TIER_BF16,
                                                     orc.TIER_UINT2, orc.TIER_UINT2]
    assert list(orc.tiers_threshold(A, 2.4, 1.9)) == [orc.TIER_BF16, orc.TIER_BF16,
                                                     orc.TIER_UINT2, orc.TIER_UINT4]


def test_tier_rank_ties_lower_channel_first():
    A = np.array([1.0, 3.0, 3.0, 1.0, 3.0], np.float32)
    assert list(orc.tiers_rank(A, 2, 2)) == [orc.TIER_UINT4, orc.TIER_BF16, orc.TIER_BF16,
                                             orc.TIER_UINT2, orc.TIER_UINT4]


def test_capped_tiers_hand_example():
    """Threshold tiers with record capacities: the overflow of a full tier
    drops one tier, smallest salience first (MixKVQ thresholds; the record
    holds at most cap_bf16 BF16 and cap_uint4 UINT4 channels)."""
    A = np.array([3.0, 1.0, 2.0, 5.0, 0.5, 2.0], np.float32)
    B, U4, U2 = orc.TIER_BF16, orc.TIER_UINT4, orc.TIER_UINT2
    # uncapped: A > 1.5 -> BF16 (d0, d2, d3, d5); 0.75 < A <= 1.5 -> UINT4 (d1)
    assert list(orc.tiers_capped(A, 1.5, 0.75, 6, 6)) == [B, U4, B, B, U2, B]
    # two BF16 slots: d3 (5.0) and d0 (3.0); d2 and d5 tie at 2.0 and drop
    # to UINT4; d1 also qualifies for UINT4
    assert list(orc.tiers_capped(A, 1.5, 0.75, 2, 6)) == [B, U4, U4, B, U2, U4]
    # two UINT4 slots as well: d2 (lower index of the tie) and d5 take them,
    # d1 (1.0) is over the UINT4 capacity -> UINT2
    assert list(orc.tiers_capped(A, 1.5, 0.75, 2, 2)) == [B, U2, U4, B, U2, U4]
    # a threshold above every A: nothing is BF16 whatever the capacity
    assert list(orc.tiers_capped(A, 9.0, 2.5, 6, 6)) == [U4, U2, U2, U4, U2, U2]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_capped_tiers_reduce_to_rank_and_threshold(seed):
    """The two special cases: thresholds at -inf give the rank rule, and
    capacities of D give the plain threshold rule."""
    rng = np.random.default_rng(seed)
    A = np.round(rng.exponential(1.0, 128), 2).astype(np.float32)   # ties included
    for nb, n4 in [(6, 25), (0, 0), (128, 0), (3, 125)]:
        assert np.array_equal(orc.tiers_capped(A, -np.inf, -np.inf, nb, n4),
                              orc.tiers_rank(A, nb, n4))
    for tb, t4 in [(1.5, 0.5), (0.2, 0.2), (9.0, 0.1), (0.5, 1.0)]:
        assert np.array_equal(orc.tiers_capped(A, tb, t4, 128, 128),
                              orc.tiers_threshold(A, tb, t4))


def test_online_accumulator_equals_window_importance():
    """MixKVQ online saliency: per-step |q| sums, divided by (n_rep * steps)
    at the window's end, give bit for bit the importance of the same window
    of queries computed in one pass."""
    rng = np.random.default_rng(4)
    n_rep, L, D = 4, 37, 128
    q = bf16_trunc(rng.standard_normal((n_rep, L, D)) * 3)
    acc = np.zeros(D, np.float32)
    for i in range(L):
        orc.observe_query(acc, q[:, i])
    I_online = orc.importance_from_sum(acc, n_rep, L)
    assert np.array_equal(I_online.view(np.uint32), orc.importance(q).view(np.uint32))


def test_mixed_cache_online_window_and_threshold_tiers():
    """A mixed cache flushed without importance takes it from the queries
    observed since the previous flush, then starts a new window; threshold
    tiers then follow tiers_capped on that importance."""
    rng = np.random.default_rng(6)
    B, Hkv, n_rep, D, R = 1, 2, 2, 128, 128
    c = orc.OracleCache(B, Hkv, D, mode="mixed", n_bf16=8, n_uint4=16,
                        tier_mode="threshold", tau_bf16=0.9, tau_uint4=0.3)
    with pytest.raises(ValueError):
        c.observe(np.zeros((B, Hkv * n_rep, 3), np.uint16))   # wrong head dim
    K = bf16_trunc(rng.standard_normal((B, Hkv, R, D)))
    V = bf16_trunc(rng.standard_normal((B, Hkv, R, D)))
    qs = [bf16_trunc(rng.standard_normal((B, Hkv * n_rep, D))) for _ in range(5)]
    for i in range(R):
        c.append(K[:, :, i], V[:, :, i])
    with pytest.raises(ValueError):
        c.flush()                                   # mixed, no importance, no window
    for q in qs:
        c.observe(q)
    want_I = orc.importance(np.stack(qs, axis=2)[0, 0:n_rep])     # unit 0's window
    c.flush()
    assert c.q_steps == 0 and not c.qacc.any()       # a new window starts
    S = orc.sensitivity(K[0, 0], 2)
    want = orc.tiers_capped(orc.salience(want_I, S), 0.9, 0.3, 8, 16)
    assert np.array_equal(c.k_groups[0][0].tiers, want)


def test_mixed_group_storage_and_reconstruction():
    G, D = 8, 6
    rng = np.random.default_rng(9)
    k = np.zeros((G, D), np.float32)
    k[:, 0] = rng.integers(0, 16, G)          # on a 4-bit grid incl. 0 and 15
    k[0, 0], k[1, 0] = 0, 15
    k[:, 1] = rng.standard_normal(G)
    k[:, 2] = [0, 1, 2, 3, 0, 1, 2, 3]        # on the 2-bit grid
    k[:, 3] = rng.standard_normal(G) * 9
    k[:, 4] = rng.standard_normal(G)
    k[:, 5] = -2.0                            # constant
    kb = orc.f32_to_bf16_exact(orc.bf16_to_f32(
        (k.view(np.uint32) >> 16).astype(np.uint16)))      # truncate to bf16 values
    tiers = np.array([orc.TIER_UINT4, orc.TIER_UINT2, orc.TIER_UINT2,
                      orc.TIER_BF16, orc.TIER_UINT4, orc.TIER_UINT2], np.uint8)
    grp = orc.quantize_k_mixed_group(kb, tiers)
    assert list(grp.perm) == [3, 0, 4, 1, 2, 5]
    assert np.array_equal(grp.raw[0], kb[:, 3])
    rec = orc.dequant_k_mixed_group(grp, G)
    kf = orc.bf16_to_f32(kb).astype(np.float64)
    assert np.array_equal(rec[:, 3], kf[:, 3])            # BF16 tier verbatim
    assert np.array_equal(rec[:, 0], kf[:, 0])            # exact 4-bit grid
    assert np.array_equal(rec[:, 2], kf[:, 2])            # exact 2-bit grid
    assert np.array_equal(rec[:, 5], kf[:, 5])            # constant channel
    assert grp.s4[1] == np.float32(np.float32(kf[:, 4].max() - kf[:, 4].min()) / np.float32(15))
    assert np.all(np.abs(rec[:, 4] - kf[:, 4]) <= grp.s4[1] * (0.5 + 2**-18))
    assert np.all(np.abs(rec[:, 1] - kf[:, 1]) <= grp.s2[0] * (0.5 + 2**-18))


# ---------------------------------------------------------- byte accounting
def test_byte_formula_example():
    g = golden("kivi_byte_formula.json")
    args = dict(T=g["T"], D=g["D"], k_bits=g["b"], v_bits=g["b"], Gk=g["G"], Gv=g["G"],
                origin_bytes=g["e"], step_bytes=g["e"])
    total = orc.cache_bytes(rK=g["rK"], rV=g["rV"], float_bytes=g["f"], **args)
    quant = orc.cache_bytes(rK=g["rK"], rV=g["rV"], float_bytes=0, **args)
    assert total == g["total_kib"] * 1024
    assert round(quant / 1024) == g["quantized_kib"]
    assert total - quant == g["residual_kib"] * 1024
    assert 2 * g["T"] * g["D"] * g["f"] == g["unquantized_mib"] * 2**20
    one = orc.cache_bytes(T=g["G"], rK=0, rV=0, D=1, k_bits=g["b"], v_bits=g["b"], Gk=g["G"],
                          Gv=g["G"], origin_bytes=g["e"], step_bytes=g["e"], float_bytes=g["f"])
    assert one * 8 / (2 * g["G"]) == g["bits_per_element"]


# ------------------------------------------------ attention-sink window (f3)
# PN-Mix keeps the first N_s = 32 tokens at original precision ahead of the
# residual buffer; InnerQ keeps a high-precision window for attention-sink
# tokens.  Reading: tokens [0, n_sink) of the sequence stay bf16 and are
# never quantized; groups and the residual follow them.

def _bf16(x):
    """bf16 bits of x truncated toward zero (any bf16 values will do)."""
    x = np.ascontiguousarray(x, np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _seq(L, seed, D=32):
    rng = np.random.default_rng(seed)
    return _bf16(rng.standard_normal((1, 1, L, D))), _bf16(rng.standard_normal((1, 1, L, D)))


def test_sink_only_cache_is_plain_bf16_attention():
    K, V = _seq(20, 1)
    q = _bf16(np.random.default_rng(2).standard_normal((1, 1, 32)))
    c = orc.OracleCache(1, 1, 32, Gk=4, R=4, n_sink=32)
    c.prefill(K, V)
    assert (c.s, c.T_q, c.r) == (20, 0, 0)
    ref = orc.attention(orc.bf16_to_f32(q[0, 0]).astype(np.float64),
                        orc.bf16_to_f32(K[0, 0]).astype(np.float64),
                        orc.bf16_to_f32(V[0, 0]).astype(np.float64))
    assert np.allclose(c.attention(q)[0, 0], ref, rtol=0, atol=1e-12)


def test_sink_shifts_quantization_by_its_length():
    K, V = _seq(3 + 9 * 4 + 2, 3)
    a = orc.OracleCache(1, 1, 32, Gk=4, R=4, n_sink=3)
    a.prefill(K, V)
    b = orc.OracleCache(1, 1, 32, Gk=4, R=4)
    b.prefill(K[:, :, 3:], V[:, :, 3:])
    assert (a.s, a.T_q, a.r) == (3, b.T_q, b.r) == (3, 36, 2)
    for (ca, ma, sa), (cb, mb, sb) in zip(a.k_groups[0], b.k_groups[0]):
        assert np.array_equal(ca, cb) and np.array_equal(ma, mb) and np.array_equal(sa, sb)
    assert np.array_equal(a.sink_k[0], K[0, 0, :3]) and np.array_equal(a.sink_v[0], V[0, 0, :3])


def test_sink_fills_before_the_residual_on_append():
    K, V = _seq(2, 4)
    c = orc.OracleCache(1, 1, 32, Gk=4, R=4, n_sink=3)
    c.prefill(K, V)
    k2, v2 = _seq(9, 5)
    lengths = []
    for i in range(9):
        c.append(k2[0, 0, i], v2[0, 0, i])
        if c.r == c.R:
            c.flush()
        lengths.append((c.s, c.T_q, c.r))
    assert lengths == [(3, 0, 0), (3, 0, 1), (3, 0, 2), (3, 0, 3), (3, 4, 0), (3, 4, 1),
                       (3, 4, 2), (3, 4, 3), (3, 8, 0)]
    assert np.array_equal(c.sink_k[0, 2], k2[0, 0, 0])


def test_sink_attention_is_attention_over_sink_then_history():
    K, V = _seq(5 + 2 * 4 + 1, 6)
    q = _bf16(np.random.default_rng(7).standard_normal((1, 1, 32)))
    a = orc.OracleCache(1, 1, 32, Gk=4, R=4, n_sink=5)
    a.prefill(K, V)
    b = orc.OracleCache(1, 1, 32, Gk=4, R=4)
    b.prefill(K[:, :, 5:], V[:, :, 5:])
    kb, vb = b.dequant_unit(0)
    ks = orc.bf16_to_f32(K[0, 0, :5]).astype(np.float64)
    vs = orc.bf16_to_f32(V[0, 0, :5]).astype(np.float64)
    ref = orc.attention(orc.bf16_to_f32(q[0, 0]).astype(np.float64),
                        np.concatenate([ks, kb]), np.concatenate([vs, vb]))
    assert np.allclose(a.attention(q)[0, 0], ref, rtol=0, atol=1e-12)


# ------------------------------------------- KIVI variant (V FIFO, G < R)
def _bf(bits):
    """The fp32 value of one bf16 bit pattern."""
    return float(orc.bf16_to_f32(np.array([bits], np.uint16))[0])


def _bf16_vec(x):
    """Nearest-even bf16 bits of an fp32 vector."""
    return np.array([orc.f32_to_bf16_rn(v) for v in np.asarray(x, np.float32)], np.uint16)


def _kivi_token(t, D):
    """Token t's key and value rows (bf16 bits), chosen so that 1-bit groups
    of two tokens (keys) or two channels (values) reconstruct exactly."""
    k = np.full(D, float(t), np.float32)
    v = np.array([t + 0.5 * (c % 2) for c in range(D)], np.float32)
    return orc.f32_to_bf16_exact(k), orc.f32_to_bf16_exact(v)


def test_kivi_trace_persisted_lengths_and_order():
    """KIVI §5's trace (R = 4, G = 2, nine tokens): key residual lengths
    1,2,3,0,1,2,3,0,1 and value residual lengths min(t, R) after every step;
    the quantized part and the residual together hold every token in order;
    at step 9 keys split 8 + 1 and values 5 + 4 (Algorithm 1 order)."""
    g = golden("kivi_residual_trace.json")
    R, G, D = g["R"], g["G"], 4
    cache = orc.KiviOracleCache(1, 1, D, k_bits=1, v_bits=1, G=G, R=R)
    kl, vl = [], []
    for t in range(1, g["steps"] + 1):
        k, v = _kivi_token(t, D)
        cache.append(k[None, None], v[None, None])
        nk, rk, nv, rv = cache.lengths()
        kl.append(rk)
        vl.append(rv)
        K, V = cache.dequant_unit(0)
        want_k = np.stack([orc.bf16_to_f32(_kivi_token(i, D)[0]) for i in range(1, t + 1)])
        want_v = np.stack([orc.bf16_to_f32(_kivi_token(i, D)[1]) for i in range(1, t + 1)])
        assert np.array_equal(K, want_k) and np.array_equal(V, want_v)
    assert kl == g["persisted_key_residual_lengths"]
    assert vl == g["persisted_value_residual_lengths"]
    nk, rk, nv, rv = cache.lengths()
    assert [nk, rk] == g["step9_key_split"] and [nv, rv] == g["step9_value_split"]


def test_kivi_prefill_leaves_the_state_of_appends():
    """A prefill of L tokens leaves what L appends leave (§5's persisted
    invariants), for every L up to three windows."""
    R, G, D = 4, 2, 4
    rng = np.random.default_rng(3)
    toks = [(_bf16_vec(rng.standard_normal(D)), _bf16_vec(rng.standard_normal(D)))
            for _ in range(13)]
    for L in range(0, 13):
        a = orc.KiviOracleCache(1, 1, D, G=G, R=R)
        for k, v in toks[:L]:
            a.append(k[None, None], v[None, None])
        b = orc.KiviOracleCache(1, 1, D, G=G, R=R)
        K = np.stack([k for k, _ in toks[:L]]).reshape(1, 1, L, D) if L else np.zeros((1, 1, 0, D), np.uint16)
        V = np.stack([v for _, v in toks[:L]]).reshape(1, 1, L, D) if L else np.zeros((1, 1, 0, D), np.uint16)
        b.prefill(K, V)
        assert a.lengths() == b.lengths()
        Ka, Va = a.dequant_unit(0)
        Kb, Vb = b.dequant_unit(0)
        assert np.array_equal(Ka, Kb) and np.array_equal(Va, Vb)


def test_kivi_value_rows_follow_the_value_boundary():
    """§6: one softmax over all visible tokens, then the probabilities meet
    the values at the values' own boundary.  At step 9 (keys 8 + 1, values
    5 + 4) the cache's attention equals textbook attention over the tokens'
    keys and values rebuilt one by one: the first 8 keys and 5 values from
    their quantized groups, the rest exact."""
    R, G, D = 4, 2, 4
    rng = np.random.default_rng(11)
    cache = orc.KiviOracleCache(1, 1, D, k_bits=2, v_bits=2, G=G, R=R)
    raw_k, raw_v = [], []
    for _ in range(9):
        k = _bf16_vec(rng.standard_normal(D))
        v = _bf16_vec(rng.standard_normal(D))
        raw_k.append(orc.bf16_to_f32(k))
        raw_v.append(orc.bf16_to_f32(v))
        cache.append(k[None, None], v[None, None])
    Kx = np.stack(raw_k).astype(np.float64)
    Vx = np.stack(raw_v).astype(np.float64)
    Kh, Vh = Kx.copy(), Vx.copy()
    for t0 in range(0, 8, G):          # keys: groups of G tokens per channel
        for d in range(D):
            c, o, s = orc.quantize_group_bf16(Kx[t0:t0 + G, d], 2)
            Kh[t0:t0 + G, d] = orc.dequantize_group(c, _bf(o),
                                                    _bf(s))
    for t in range(5):                 # values: groups of G channels per token
        for j in range(0, D, G):
            c, o, s = orc.quantize_group_bf16(Vx[t, j:j + G], 2)
            Vh[t, j:j + G] = orc.dequantize_group(c, _bf(o),
                                                  _bf(s))
    q = _bf16_vec(rng.standard_normal(D))
    got = cache.attention(q[None, None])[0, 0]
    qf = orc.bf16_to_f32(q).astype(np.float64)
    s = Kh @ qf / np.sqrt(D)
    p = np.exp(s - s.max())
    want = (p / p.sum()) @ Vh
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # taking the first 8 value rows from quantized groups (the key boundary)
    # would give another output
    Vw = Vx.copy()
    for t in range(8):
        for j in range(0, D, G):
            c, o, s2 = orc.quantize_group_bf16(Vx[t, j:j + G], 2)
            Vw[t, j:j + G] = orc.dequantize_group(c, _bf(o),
                                                  _bf(s2))
    assert np.max(np.abs((p / p.sum()) @ Vw - want)) > 1e-6


def test_kivi_bf16_metadata_key_example():
    """§3's 4x4 Key example with §7's metadata in the input dtype (bf16):
    the per-token row 0 keeps the page's codes [3, 0, 0, 0] with the bf16
    step bf16(101/3) = 33.75, so its top value rebuilds as -1 + 3 * 33.75 =
    100.25 instead of the page's 100; per channel the steps 1 and 1/2 are
    exact in bf16 and the columns rebuild exactly."""
    g = golden("kivi_key_4x4.json")
    codes, o, s = orc.quantize_group_bf16(g["key"][0], g["bits"])
    assert list(codes) == [3, 0, 0, 0]
    assert _bf(o) == -1.0
    assert _bf(s) == 33.75
    assert abs(Fraction(33.75) - frac(g["per_token_row0_step"])) <= Fraction(1, 2**8) * 101 / 3
    rec = orc.dequantize_group(codes, -1.0, 33.75)
    assert rec[0] == 100.25 and list(rec[1:]) == [-1.0, -1.0, -1.0]
    for col in range(4):
        column = [r[col] for r in g["key"]]
        c, o, s = orc.quantize_group_bf16(column, 2)
        rec = orc.dequantize_group(c, _bf(o), _bf(s))
        assert np.array_equal(rec, np.asarray(column, np.float64))


def test_kivi_bf16_quantizer_special_cases_and_bound():
    """Constant group: step 0, codes 0, exact.  RNE ties where bf16 is exact
    ([0, 0.5, 2.5, 3] -> [0, 0, 2, 3]).  A hand-worked group where the bf16
    rounding of x - m decides a code.  On random bf16 groups the error
    stays within 0.52 steps: the bf16 roundings of x - m and of the quotient
    move a 2-bit quotient by at most 3 * 2^-8 (< 0.012), and 3 bf16 steps
    stay within 2^-8 of the range."""
    c, o, s = orc.quantize_group_bf16([2.5] * 7, 2)
    assert list(c) == [0] * 7 and s == 0 and _bf(o) == 2.5
    c, o, s = orc.quantize_group_bf16([0.0, 0.5, 2.5, 3.0], 2)
    assert list(c) == [0, 0, 2, 3]
    # x - m is rounded to bf16 before the division: m = -2^-7, M = 2.5 give
    # R = bf16(2.5078125) = 2.5 (a tie, to even) and step = bf16(2.5 / 3) =
    # 0.83203125; for x = 2.078125, x - m = 2.0859375 rounds (a tie) to
    # 2.09375 and bf16(2.09375 / 0.83203125) = 2.515625 gives code 3, where
    # the unrounded difference would give the quotient 2.5 and code 2.
    c, o, s = orc.quantize_group_bf16([-2.0 ** -7, 2.078125, 2.5], 2)
    assert _bf(s) == 0.83203125 and list(c) == [0, 3, 3]
    rng = np.random.default_rng(5)
    worst = 0.0
    for _ in range(300):
        x = rng.standard_normal(32).astype(np.float32) * rng.choice([1e-3, 1.0, 50.0])
        x = orc.bf16_to_f32(_bf16_vec(x))
        c, o, s = orc.quantize_group_bf16(x, 2)
        step = _bf(s)
        rec = orc.dequantize_group(c, _bf(o), step)
        worst = max(worst, float(np.max(np.abs(rec - x.astype(np.float64)))) / step)
    assert worst <= 0.52


# ------------------------------------------------------ PN-Mix H3/L1 (f4)
def _bf16_of(x):
    """Nearest-even bf16 bits of an fp32 array (any shape)."""
    x = np.asarray(x, np.float32)
    return np.array([orc.f32_to_bf16_rn(v) for v in x.reshape(-1)], np.uint16).reshape(x.shape)

def test_pnmix_eq7_one_bit_groups_rebuild_at_quarter_points():
    """PN-Mix Eq. 7: s = (max - min)/2, z = (3 min + max)/4, so the two
    reconstructions are the quarter points (3m + M)/4 and (m + 3M)/4; codes
    split at the midpoint (a tie at the midpoint rounds to even, code 0);
    a constant group has zero scale and the original offset; the error is
    at most a quarter of the range."""
    c, z, s = orc.quantize_group_1bit_mid([0.0, 1.0, 3.0, 4.0])
    assert list(c) == [0, 0, 1, 1] and z == 1.0 and s == 2.0
    assert sorted({float(z), float(z + s)}) == [(3 * 0 + 4) / 4, (0 + 3 * 4) / 4]
    c, z, s = orc.quantize_group_1bit_mid([0.0, 2.0, 4.0])
    assert list(c) == [0, 0, 1]
    c, z, s = orc.quantize_group_1bit_mid([-1.5] * 5)
    assert list(c) == [0] * 5 and z == -1.5 and s == 0.0
    rng = np.random.default_rng(8)
    for _ in range(200):
        x = (rng.standard_normal(128) * rng.choice([1e-2, 1.0, 30.0])).astype(np.float32)
        c, z, s = orc.quantize_group_1bit_mid(x)
        rec = np.float64(z) + np.float64(s) * c
        quarter = (float(x.max()) - float(x.min())) / 4
        assert np.max(np.abs(rec - x)) <= quarter * (1 + 2 ** -20)


def test_pnmix_eq7_codes_brute_force_nearest():
    """Eq. 7 by brute force: each 1-bit code selects the nearer of its
    group's two reconstruction points z and z + s (exact rationals), the
    lower one at an exact tie."""
    rng = np.random.default_rng(77)
    for trial in range(300):
        n = int(rng.integers(2, 9))
        x = (rng.integers(-40, 40, n) / rng.choice([1, 2, 4, 8])).astype(np.float32)
        if trial % 3 == 0:
            x = rng.standard_normal(n).astype(np.float32)
        if x.max() == x.min():
            continue
        c, z, s = orc.quantize_group_1bit_mid(x)
        Z, S = Fraction(float(z)), Fraction(float(s))
        for xi, ci in zip(x, c):
            X = Fraction(float(xi))
            d = [abs(X - Z), abs(X - Z - S)]
            if d[0] == d[1]:
                assert ci == 0
            else:
                # fp32 (x - z) / s rounds twice: a code may differ only at a
                # near tie
                assert d[int(ci)] <= min(d) + S * Fraction(1, 2**20)


def test_pnmix_eq6_pair_scores_by_hand():
    """PN-Mix Eq. 6 on integer pair norms: two query heads of one GQA group,
    two tokens each, two keys, D = 4 (adjacent pairs (0,1), (2,3)).  Query
    pair norms: head 0 pair 0 -> 5, 10 (mean 7.5), pair 1 -> 0, 1 (0.5);
    head 1 pair 0 -> 0, 0, pair 1 -> 5, 0 (2.5); head averages 3.75, 1.5.
    Key pair norms 1, 1 and 2, 0: means 1 and 1.  sigma = [3.75, 1.5].  The
    split layout pairs (i, i + D/2): the same scores as the adjacent layout
    on channels reordered [0, 2, 1, 3]."""
    bf = lambda a: orc.f32_to_bf16_exact(np.asarray(a, np.float32))
    q = bf([[[3, 4, 0, 0], [6, 8, 1, 0]], [[0, 0, 3, 4], [0, 0, 0, 0]]])
    k = bf([[1, 0, 0, 2], [0, 1, 0, 0]])
    sig = orc.pair_scores(q, k, orc.PAIR_ADJACENT)
    assert list(sig) == [3.75, 1.5]
    perm = [0, 2, 1, 3]
    assert np.array_equal(orc.pair_scores(q, k, orc.PAIR_SPLIT),
                          orc.pair_scores(q[..., perm], k[..., perm], orc.PAIR_ADJACENT))


def test_pnmix_selection_takes_whole_pairs():
    """floor(r d / 2) pairs at r = 0.5, d = 128: 32 pairs, both channels of
    each high; ties go to the lower pair index."""
    sig = np.ones(64, np.float32)
    sig[[5, 40]] = 2.0
    mask = orc.select_pairs(sig, int(0.5 * 128 // 2))
    assert mask.sum() == 32 and mask[5] and mask[40] and mask[:30].sum() == 30
    for layout in (orc.PAIR_ADJACENT, orc.PAIR_SPLIT):
        ch = orc.channel_mask(mask, layout)
        a, b = orc.pair_channels(128, layout)
        assert ch.sum() == 64 and np.array_equal(ch[a], ch[b]) and np.array_equal(ch[a], mask)


def test_pnmix_h3l1_planes_and_storage():
    """App. G: every channel keeps its code's LSB; high channels add the two
    upper bits of their 3-bit code (Eq. 2).  The main configuration (b_H = 3,
    b_L = 1, r = 0.5, G = N = 128, N_s = 32) costs about 2.26 key bits per
    element at 32K quantized tokens (PN-Mix App. G figure), here 2 (planes)
    + 0.25 (an fp16 offset and scale per channel and group) + the sink and
    the pair mask = 2.2656; without the sink it would be 2.25."""
    rng = np.random.default_rng(9)
    kg = _bf16_of(rng.standard_normal((128, 16)))
    high = np.zeros(16, bool)
    high[[0, 1, 6, 7]] = True
    codes, off, sc = orc.quantize_k_h3l1_group(kg, high)
    lsb, upper = orc.h3l1_planes(codes, high)
    assert upper.shape == (128, 4) and lsb.shape == (128, 16)
    assert np.array_equal((upper << 1) | lsb[:, high], codes[:, high])
    assert codes[:, ~high].max() <= 1 and codes[:, high].max() <= 7
    x = orc.bf16_to_f32(kg)
    for d in np.flatnonzero(high):   # Eq. 2 at 3 bits: |x - x^| <= s/2
        rec = np.float64(off[d]) + np.float64(sc[d]) * codes[:, d]
        assert np.max(np.abs(rec - x[:, d])) <= float(sc[d]) / 2 * (1 + 2 ** -20)
    bits = orc.pnmix_k_bits(32768, 128, 128, 32, 32)
    assert abs(bits - 2.26) < 0.006
    assert abs(orc.pnmix_k_bits(32768, 128, 128, 32, 0) - 2.26) >= 0.006


def test_pnmix_cache_attention_over_rebuilt_keys():
    """A PN-Mix cache (the pair mask fixed before prefill; keys by H3/L1 per
    128-token group, values as the main path) attends like textbook
    attention over keys rebuilt group by group."""
    rng = np.random.default_rng(12)
    D, L = 8, 2 * 128 + 20
    K = _bf16_of(rng.standard_normal((1, 1, L, D)))
    V = _bf16_of(rng.standard_normal((1, 1, L, D)))
    high = np.zeros((1, 1, D), bool)
    high[0, 0, [2, 3]] = True
    cache = orc.OracleCache(1, 1, D, k_bits=2, v_bits=2, Gk=128, Gv=4, R=128, mode="pnmix",
                            high_channels=high)
    cache.prefill(K, V)
    Kh = orc.bf16_to_f32(K[0, 0]).astype(np.float64)
    for g0 in (0, 128):
        codes, off, sc = orc.quantize_k_h3l1_group(K[0, 0, g0:g0 + 128], high[0, 0])
        Kh[g0:g0 + 128] = off[None, :].astype(np.float64) + sc[None, :].astype(np.float64) * codes
    _, Vh = cache.dequant_unit(0)
    q = _bf16_of(rng.standard_normal((1, 1, D)))
    got = cache.attention(q)[0, 0]
    qf = orc.bf16_to_f32(q[0, 0]).astype(np.float64)
    s = Kh @ qf / np.sqrt(D)
    p = np.exp(s - s.max())
    np.testing.assert_allclose(got, (p / p.sum()) @ Vh, rtol=1e-12, atol=1e-12)
