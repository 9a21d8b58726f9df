"""Plain CPU oracle for low-bit KV-cache quantization and decode attention.

TEST INFRASTRUCTURE ONLY.  The product library (``bit_kv_cache_kvq_gb300``)
never imports, loads or calls anything here; only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` do.  The
numeric work lives in ``kvq_oracle.c`` (single-threaded, fp32 quantization
with IEEE division and round-half-to-even codes, fp64 attention); this module
marshals numpy arrays into it and walks the cache state machine of MixKVQ's
Algorithm 1 (prefill split, append, flush when the residual is full).

bf16 arrays are numpy ``uint16`` arrays of raw bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

ORC_OK, ORC_ERR_ARG, ORC_ERR_NONFINITE, ORC_ERR_RANGE = 0, 1, 2, 3
TIER_BF16, TIER_UINT4, TIER_UINT2 = 0, 1, 2


class OracleError(ValueError):
    """A group or call the pages' validation rules reject."""

    def __init__(self, status: int, what: str):
        names = {ORC_ERR_ARG: "ARG", ORC_ERR_NONFINITE: "NONFINITE",
                 ORC_ERR_RANGE: "RANGE"}
        super().__init__(f"{what}: {names.get(status, status)}")
        self.status = status


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into liboracle.so beside it (gcc, no fast-math,
    no floating-point contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fno-strict-aliasing", "-Wall", "-Wextra",
           "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i, l, f, d = ctypes.c_int, ctypes.c_long, ctypes.c_float, ctypes.c_double
        sig = {
            "orc_quantize_group": (i, [P, l, l, i, P, P, P]),
            "orc_quantize_group_bf16": (i, [P, l, l, i, P, P, P]),
            "orc_f32_to_bf16_rn": (ctypes.c_uint16, [f]),
            "orc_quantize_group_1bit_mid": (i, [P, l, l, P, P, P]),
            "orc_pair_scores": (i, [P, i, i, P, i, i, i, P]),
            "orc_pack_lsb": (None, [P, l, i, P]),
            "orc_unpack_lsb": (None, [P, l, i, P]),
            "orc_quantize_k_unit": (i, [P, l, i, i, i, P, P, P]),
            "orc_quantize_v_unit": (i, [P, l, i, i, i, P, P, P]),
            "orc_dequant_k_unit": (None, [P, P, P, l, i, i, i, P]),
            "orc_dequant_v_unit": (None, [P, P, P, l, i, i, i, P]),
            "orc_attention": (i, [P, P, P, l, i, P, P]),
            "orc_importance": (i, [P, i, i, i, P]),
            "orc_sensitivity": (i, [P, i, i, i, P]),
            "orc_salience": (None, [P, P, i, P]),
            "orc_tiers_rank": (i, [P, i, i, i, P]),
            "orc_tiers_threshold": (i, [P, i, f, f, P]),
            "orc_tiers_capped": (i, [P, i, f, f, i, i, P]),
            "orc_observe_query": (i, [P, P, i, i]),
            "orc_importance_from_sum": (i, [P, i, i, i, P]),
            "orc_quantize_k_mixed_group": (i, [P, i, i, P, P, P, P, P, P, P, P, P]),
            "orc_dequant_k_mixed_group": (None, [i, i, P, i, i, P, P, P, P, P, P, P, P]),
            "orc_cache_bytes": (d, [l, l, l, i, i, i, i, i, i, i, i]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(status: int, what: str):
    if status != ORC_OK:
        raise OracleError(status, what)


# ----------------------------------------------------------------- primitives
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 patterns to fp32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_exact(x: np.ndarray) -> np.ndarray:
    """Raw bf16 pattern of fp32 values that are bf16-representable."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value is not representable in bf16")
    return (u >> 16).astype(np.uint16)


def quantize_group(x, bits: int):
    """One group: returns (codes uint8, origin fp32, step fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.size, np.uint8)
    m, s = ctypes.c_float(), ctypes.c_float()
    _check(lib().orc_quantize_group(_p(x), x.size, 1, bits, _p(codes),
                                    ctypes.byref(m), ctypes.byref(s)), "quantize_group")
    return codes, np.float32(m.value), np.float32(s.value)


def quantize_group_bf16(x, bits: int):
    """One group with bf16 metadata and bf16 arithmetic (KIVI §7): returns
    (codes uint8, origin bf16 bits, step bf16 bits)."""
    x = np.ascontiguousarray(x, np.float32).reshape(-1)
    codes = np.zeros(x.size, np.uint8)
    o, st = ctypes.c_uint16(), ctypes.c_uint16()
    _check(lib().orc_quantize_group_bf16(_p(x), x.size, 1, bits, _p(codes), ctypes.byref(o),
                                         ctypes.byref(st)), "quantize_group_bf16")
    return codes, o.value, st.value


def f32_to_bf16_rn(x: float) -> int:
    """Nearest-even bf16 bits of a finite fp32 value."""
    return int(lib().orc_f32_to_bf16_rn(float(np.float32(x))))


def quantize_group_1bit_mid(x):
    """PN-Mix Eq. 7 one-bit group: (codes, offset z, scale s), fp32."""
    x = np.ascontiguousarray(x, np.float32).reshape(-1)
    codes = np.zeros(x.size, np.uint8)
    z, sc = ctypes.c_float(), ctypes.c_float()
    _check(lib().orc_quantize_group_1bit_mid(_p(x), x.size, 1, _p(codes), ctypes.byref(z),
                                             ctypes.byref(sc)), "quantize_group_1bit_mid")
    return codes, np.float32(z.value), np.float32(sc.value)


PAIR_ADJACENT, PAIR_SPLIT = 0, 1


def pair_channels(D: int, layout: int):
    """The two channels of each RoPE pair: (2i, 2i+1) adjacent (the paper's
    formula) or (i, i + D/2) split halves (Hugging Face Llama layout)."""
    P = D // 2
    i = np.arange(P)
    return (2 * i, 2 * i + 1) if layout == PAIR_ADJACENT else (i, i + P)


def pair_scores(q_group: np.ndarray, k: np.ndarray, layout: int = PAIR_ADJACENT) -> np.ndarray:
    """PN-Mix Eq. 6: sigma [D/2] fp32 of one KV head from its GQA group's
    prefill queries (bf16 bits [Hg, Lq, D]) and keys (bf16 bits [Lk, D])."""
    q = np.ascontiguousarray(q_group, np.uint16)
    kk = np.ascontiguousarray(k, np.uint16)
    Hg, Lq, D = q.shape
    sigma = np.zeros(D // 2, np.float32)
    _check(lib().orc_pair_scores(_p(q), Hg, Lq, _p(kk), kk.shape[0], D, layout, _p(sigma)),
           "pair_scores")
    return sigma


def select_pairs(sigma: np.ndarray, n_high: int) -> np.ndarray:
    """The n_high pairs of largest sigma (ties: lower pair index) as a
    boolean pair mask."""
    order = sorted(range(sigma.size), key=lambda i: (-float(sigma[i]), i))
    mask = np.zeros(sigma.size, bool)
    mask[order[:n_high]] = True
    return mask


def channel_mask(pair_mask: np.ndarray, layout: int = PAIR_ADJACENT) -> np.ndarray:
    """Per-channel high-precision flags: both channels of a selected pair."""
    D = 2 * pair_mask.size
    a, b = pair_channels(D, layout)
    m = np.zeros(D, bool)
    m[a[pair_mask]] = True
    m[b[pair_mask]] = True
    return m


def quantize_k_h3l1_group(k_group: np.ndarray, high: np.ndarray, b_high: int = 3):
    """PN-Mix H3/L1 key group (bf16 bits [G, D]): channels with high set at
    b_high bits by Eq. 2 (min-max, origin the minimum), the others at one
    bit by Eq. 7.  Returns (codes [G, D], offset [D] fp32, scale [D] fp32)."""
    x = bf16_to_f32(np.asarray(k_group, np.uint16))
    G, D = x.shape
    codes = np.zeros((G, D), np.uint8)
    off = np.zeros(D, np.float32)
    sc = np.zeros(D, np.float32)
    for d in range(D):
        if high[d]:
            codes[:, d], off[d], sc[d] = quantize_group(x[:, d], b_high)
        else:
            codes[:, d], off[d], sc[d] = quantize_group_1bit_mid(x[:, d])
    return codes, off, sc


def h3l1_planes(codes: np.ndarray, high: np.ndarray):
    """App. G packing planes: the LSB of every code (all channels) and the
    upper two bits of the high channels' 3-bit codes."""
    return codes & 1, (codes >> 1)[:, high]


def pnmix_k_bits(T: int, D: int, G: int, n_high_pairs: int, n_sink: int,
                 meta_bits: int = 16) -> float:
    """Persistent key bits per quantized element: an LSB plane over all
    channels, two upper bits for the high channels, an offset and a scale
    per channel and group, the pair mask once, the sink tokens raw."""
    bits = T * D + T * 2 * (2 * n_high_pairs) + (T // G) * D * 2 * meta_bits
    bits += D // 2 + n_sink * D * 16
    return bits / (T * D)


def dequantize_group(codes, origin, step) -> np.ndarray:
    """x^ = m + step*c in fp64."""
    return float(origin) + float(step) * np.asarray(codes, np.float64)


def pack_lsb(codes, bits: int) -> bytes:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros((codes.size * bits + 7) // 8, np.uint8)
    lib().orc_pack_lsb(_p(codes), codes.size, bits, _p(out))
    return out.tobytes()


def unpack_lsb(packed: bytes, length: int, bits: int) -> np.ndarray:
    data = np.frombuffer(bytes(packed), np.uint8).copy()
    if not 0 <= length <= data.size * (8 // bits):
        raise ValueError("invalid logical length")
    out = np.zeros(length, np.uint8)
    lib().orc_unpack_lsb(_p(data), length, bits, _p(out))
    return out


def attention(q, k, v, p_out: bool = False):
    """fp64 decode attention of one query over rows k, v ([n, D])."""
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    n, D = k.shape
    o = np.zeros(D, np.float64)
    p = np.zeros(n, np.float64)
    _check(lib().orc_attention(_p(q), _p(k), _p(v), n, D, _p(o), _p(p)), "attention")
    return (o, p) if p_out else o


def importance(q_group: np.ndarray) -> np.ndarray:
    """q_group: bf16 bits [n_rep, Lq, D] -> I fp32 [D]."""
    q_group = np.ascontiguousarray(q_group, np.uint16)
    n_rep, Lq, D = q_group.shape
    out = np.zeros(D, np.float32)
    _check(lib().orc_importance(_p(q_group), n_rep, Lq, D, _p(out)), "importance")
    return out


def sensitivity(k_group: np.ndarray, bits: int = 2) -> np.ndarray:
    """k_group: bf16 bits [G, D] -> S fp32 [D]."""
    k_group = np.ascontiguousarray(k_group, np.uint16)
    G, D = k_group.shape
    out = np.zeros(D, np.float32)
    _check(lib().orc_sensitivity(_p(k_group), G, D, bits, _p(out)), "sensitivity")
    return out


def salience(I: np.ndarray, S: np.ndarray) -> np.ndarray:
    I = np.ascontiguousarray(I, np.float32)
    S = np.ascontiguousarray(S, np.float32)
    out = np.zeros(I.size, np.float32)
    lib().orc_salience(_p(I), _p(S), I.size, _p(out))
    return out


def tiers_rank(A: np.ndarray, n_bf16: int, n_uint4: int) -> np.ndarray:
    A = np.ascontiguousarray(A, np.float32)
    out = np.zeros(A.size, np.uint8)
    _check(lib().orc_tiers_rank(_p(A), A.size, n_bf16, n_uint4, _p(out)), "tiers_rank")
    return out


def tiers_threshold(A: np.ndarray, tau_bf16: float, tau_uint4: float) -> np.ndarray:
    A = np.ascontiguousarray(A, np.float32)
    out = np.zeros(A.size, np.uint8)
    _check(lib().orc_tiers_threshold(_p(A), A.size, tau_bf16, tau_uint4, _p(out)),
           "tiers_threshold")
    return out


def tiers_capped(A: np.ndarray, tau_bf16: float, tau_uint4: float, cap_bf16: int,
                 cap_uint4: int) -> np.ndarray:
    """Threshold tiers with at most cap_bf16 BF16 and cap_uint4 UINT4
    channels, taken from the largest A down (kvq_oracle.c orc_tiers_capped)."""
    A = np.ascontiguousarray(A, np.float32)
    out = np.zeros(A.size, np.uint8)
    _check(lib().orc_tiers_capped(_p(A), A.size, tau_bf16, tau_uint4, cap_bf16, cap_uint4,
                                  _p(out)), "tiers_capped")
    return out


def observe_query(acc: np.ndarray, q_step: np.ndarray) -> None:
    """acc fp32 [D] += |q| of each head row of q_step (bf16 bits [n_rep, D]),
    heads in order (MixKVQ online saliency accumulator)."""
    q_step = np.ascontiguousarray(q_step, np.uint16)
    assert acc.dtype == np.float32 and acc.flags["C_CONTIGUOUS"]
    n_rep, D = q_step.shape
    _check(lib().orc_observe_query(_p(acc), _p(q_step), n_rep, D), "observe_query")


def importance_from_sum(acc: np.ndarray, n_rep: int, steps: int) -> np.ndarray:
    acc = np.ascontiguousarray(acc, np.float32)
    out = np.zeros(acc.size, np.float32)
    _check(lib().orc_importance_from_sum(_p(acc), n_rep, steps, acc.size, _p(out)),
           "importance_from_sum")
    return out


def cache_bytes(T, rK, rV, D, k_bits, v_bits, Gk, Gv, origin_bytes, step_bytes,
                float_bytes) -> float:
    return lib().orc_cache_bytes(T, rK, rV, D, k_bits, v_bits, Gk, Gv,
                                 origin_bytes, step_bytes, float_bytes)


# ------------------------------------------------------------ unit-level parts
def quantize_k_unit(k: np.ndarray, G: int, bits: int):
    """k bf16 [T, D] -> (codes [T/G, D, ceil(G*bits/8)], kmin bf16 [T/G, D], kscale)."""
    k = np.ascontiguousarray(k, np.uint16)
    T, D = k.shape
    codes = np.zeros((T // G, D, (G * bits + 7) // 8), np.uint8)
    kmin = np.zeros((T // G, D), np.uint16)
    kscale = np.zeros((T // G, D), np.float32)
    _check(lib().orc_quantize_k_unit(_p(k), T, D, G, bits, _p(codes), _p(kmin),
                                     _p(kscale)), "quantize_k_unit")
    return codes, kmin, kscale


def quantize_v_unit(v: np.ndarray, G: int, bits: int):
    """v bf16 [T, D] -> (codes [T, D*bits/8], vmin bf16 [T, D/G], vscale)."""
    v = np.ascontiguousarray(v, np.uint16)
    T, D = v.shape
    codes = np.zeros((T, D * bits // 8), np.uint8)
    vmin = np.zeros((T, D // G), np.uint16)
    vscale = np.zeros((T, D // G), np.float32)
    _check(lib().orc_quantize_v_unit(_p(v), T, D, G, bits, _p(codes), _p(vmin),
                                     _p(vscale)), "quantize_v_unit")
    return codes, vmin, vscale


def dequant_k_unit(codes, kmin, kscale, G: int, bits: int) -> np.ndarray:
    n_groups, D, _ = codes.shape
    T = n_groups * G
    out = np.zeros((T, D), np.float64)
    if T:
        lib().orc_dequant_k_unit(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(kmin)),
                                 _p(np.ascontiguousarray(kscale)), T, D, G, bits, _p(out))
    return out


def dequant_v_unit(codes, vmin, vscale, G: int, bits: int) -> np.ndarray:
    T = codes.shape[0]
    D = codes.shape[1] * 8 // bits
    out = np.zeros((T, D), np.float64)
    if T:
        lib().orc_dequant_v_unit(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(vmin)),
                                 _p(np.ascontiguousarray(vscale)), T, D, G, bits, _p(out))
    return out


@dataclass
class MixedGroup:
    """One mixed-precision key group in canonical form."""
    tiers: np.ndarray   # uint8 [D]
    perm: np.ndarray    # uint8 [D]
    raw: np.ndarray     # uint16 [n_bf16, G]
    c4: np.ndarray      # uint8 [n_uint4, G/2]
    m4: np.ndarray      # uint16 [n_uint4]
    s4: np.ndarray      # fp32 [n_uint4]
    c2: np.ndarray      # uint8 [n_uint2, G/4]
    m2: np.ndarray      # uint16 [n_uint2]
    s2: np.ndarray      # fp32 [n_uint2]


def quantize_k_mixed_group(k_group: np.ndarray, tiers: np.ndarray) -> MixedGroup:
    k_group = np.ascontiguousarray(k_group, np.uint16)
    tiers = np.ascontiguousarray(tiers, np.uint8)
    G, D = k_group.shape
    nb = int((tiers == TIER_BF16).sum())
    n4 = int((tiers == TIER_UINT4).sum())
    n2 = D - nb - n4
    g = MixedGroup(tiers.copy(), np.zeros(D, np.uint8), np.zeros((nb, G), np.uint16),
                   np.zeros((n4, G // 2), np.uint8), np.zeros(n4, np.uint16),
                   np.zeros(n4, np.float32), np.zeros((n2, G // 4), np.uint8),
                   np.zeros(n2, np.uint16), np.zeros(n2, np.float32))
    _check(lib().orc_quantize_k_mixed_group(
        _p(k_group), G, D, _p(tiers), _p(g.perm), _p(g.raw), _p(g.c4), _p(g.m4),
        _p(g.s4), _p(g.c2), _p(g.m2), _p(g.s2)), "quantize_k_mixed_group")
    return g


def dequant_k_mixed_group(g: MixedGroup, G: int) -> np.ndarray:
    D = g.perm.size
    out = np.zeros((G, D), np.float64)
    lib().orc_dequant_k_mixed_group(G, D, _p(g.perm), g.raw.shape[0], g.c4.shape[0],
                                    _p(g.raw), _p(g.c4), _p(g.m4), _p(g.s4), _p(g.c2),
                                    _p(g.m2), _p(g.s2), _p(out))
    return out


# ------------------------------------------------------------- state machine
class OracleCache:
    """Per-layer cache walked as in MixKVQ Algorithm 1 (block flush of K and V
    together when the residual holds R tokens; prefill keeps L mod R tokens
    in the residual).  Holds canonical arrays per (batch row, KV head).

    mode "uniform": K k_bits per channel over Gk tokens; V v_bits per token
    over Gv channels.  mode "mixed": K tiers per flushed group from
    A = I * S (S at sal_bits), V as in uniform; tier_mode "rank" takes the
    n_bf16 largest A as BF16 and the next n_uint4 as UINT4, tier_mode
    "threshold" applies tau_bf16 / tau_uint4 with n_bf16 / n_uint4 as the
    group's capacities (tiers_capped).

    Online saliency (MixKVQ "efficient online salience estimation"): observe
    adds each decode step's |q| to a running sum per (unit, channel); a mixed
    flush given no importance takes I_d = sum / (n_rep * steps) over the
    steps observed since the previous flush, then starts a new window.

    n_sink > 0: the first n_sink tokens of the sequence are attention sinks
    kept in bf16 and never quantized (PN-Mix "sink 原精度保护", N_s = 32;
    InnerQ's high-precision window for attention-sink tokens).  The
    quantized groups and the residual start after them; while the sink is
    not full, appended tokens go to it.
    """

    def __init__(self, B, Hkv, D, k_bits=2, v_bits=2, Gk=128, Gv=32, R=128,
                 mode="uniform", n_bf16=0, n_uint4=0, sal_bits=2, n_sink=0,
                 tier_mode="rank", tau_bf16=0.0, tau_uint4=0.0, high_channels=None):
        if R % Gk:
            raise ValueError("R must be a multiple of the key group")
        self.B, self.Hkv, self.D = B, Hkv, D
        self.k_bits, self.v_bits, self.Gk, self.Gv, self.R = k_bits, v_bits, Gk, Gv, R
        self.mode, self.n_bf16, self.n_uint4, self.sal_bits = mode, n_bf16, n_uint4, sal_bits
        if tier_mode not in ("rank", "threshold"):
            raise ValueError("tier_mode is 'rank' or 'threshold'")
        self.tier_mode, self.tau_bf16, self.tau_uint4 = tier_mode, tau_bf16, tau_uint4
        # mode "pnmix": high_channels [B, Hkv, D] bool, the PN-Mix pair mask
        # chosen once at prefill (channel_mask of select_pairs of pair_scores)
        self.high = None if high_channels is None else np.asarray(high_channels, bool)
        if mode == "pnmix" and self.high is None:
            raise ValueError("pnmix mode needs the high-precision channels")
        U = B * Hkv
        self.qacc = np.zeros((U, D), np.float32)   # online |q| sums of the window
        self.q_steps = 0
        self.q_rep = 0
        self.k_groups = [[] for _ in range(U)]   # uniform: (codes, kmin, kscale) per group
        self.v_parts = [[] for _ in range(U)]    # (codes, vmin, vscale) per token block
        self.res_k = np.zeros((U, R, D), np.uint16)
        self.res_v = np.zeros((U, R, D), np.uint16)
        self.n_sink = n_sink
        self.sink_k = np.zeros((U, n_sink, D), np.uint16)
        self.sink_v = np.zeros((U, n_sink, D), np.uint16)
        self.s = 0
        self.T_q = 0
        self.r = 0

    # -- Algorithm 1, Prefill: r = l_prompt mod R (F read as 0)
    def prefill(self, K: np.ndarray, V: np.ndarray, importance: np.ndarray | None = None):
        if self.T_q or self.r or self.s:
            raise ValueError("prefill into a non-empty cache")
        s = min(K.shape[2], self.n_sink)
        if s:   # the sink takes the first tokens; the rest follows Algorithm 1
            for u in range(self.B * self.Hkv):
                b, h = divmod(u, self.Hkv)
                self.sink_k[u, :s] = K[b, h, :s]
                self.sink_v[u, :s] = V[b, h, :s]
            self.s = s
            K, V = K[:, :, s:], V[:, :, s:]
        B, Hkv, L, D = K.shape
        r = L % self.R
        n_q = L - r
        for u in range(B * Hkv):
            b, h = divmod(u, Hkv)
            for g0 in range(0, n_q, self.R):
                self._flush_block(u, K[b, h, g0:g0 + self.R], V[b, h, g0:g0 + self.R],
                                  None if importance is None else importance[b, h])
            self.res_k[u, :r] = K[b, h, n_q:]
            self.res_v[u, :r] = V[b, h, n_q:]
        self.T_q, self.r = n_q, r

    # -- Algorithm 1, Decoding: append to the residual
    def append(self, k_new: np.ndarray, v_new: np.ndarray):
        if self.s < self.n_sink:   # the sequence's first tokens fill the sink
            self.sink_k[:, self.s] = k_new.reshape(-1, self.D)
            self.sink_v[:, self.s] = v_new.reshape(-1, self.D)
            self.s += 1
            return
        if self.r == self.R:
            raise ValueError("residual full: flush first")
        self.res_k[:, self.r] = k_new.reshape(-1, self.D)
        self.res_v[:, self.r] = v_new.reshape(-1, self.D)
        self.r += 1

    # -- online saliency: one decode step's query (bf16 bits [B, Hq, D])
    def observe(self, q: np.ndarray):
        B, Hq, D = q.shape
        if B != self.B or D != self.D or Hq % self.Hkv:
            raise ValueError("query shape does not match the cache")
        n_rep = Hq // self.Hkv
        if self.q_steps and n_rep != self.q_rep:
            raise ValueError("query heads changed within a window")
        for u in range(self.B * self.Hkv):
            b, h = divmod(u, self.Hkv)
            observe_query(self.qacc[u], q[b, h * n_rep:(h + 1) * n_rep])
        self.q_rep = n_rep
        self.q_steps += 1

    def window_importance(self) -> np.ndarray:
        """I [B, Hkv, D] of the queries observed since the last flush."""
        if self.q_steps == 0:
            raise ValueError("no query observed in this window")
        I = np.stack([importance_from_sum(self.qacc[u], self.q_rep, self.q_steps)
                      for u in range(self.B * self.Hkv)])
        return I.reshape(self.B, self.Hkv, self.D)

    # -- Algorithm 1, Decoding: when len == R, quantize K and V, empty residual
    def flush(self, importance: np.ndarray | None = None):
        if self.r != self.R:
            raise ValueError("flush needs a full residual")
        if self.mode == "mixed" and importance is None:   # the online window
            importance = self.window_importance()
            self.qacc[:] = 0.0
            self.q_steps = 0
        for u in range(self.B * self.Hkv):
            b, h = divmod(u, self.Hkv)
            self._flush_block(u, self.res_k[u], self.res_v[u],
                              None if importance is None else importance[b, h])
        self.T_q += self.R
        self.r = 0

    def _flush_block(self, u, kb, vb, imp):
        for g0 in range(0, self.R, self.Gk):
            kg = kb[g0:g0 + self.Gk]
            if self.mode == "uniform":
                self.k_groups[u].append(quantize_k_unit(kg, self.Gk, self.k_bits))
            elif self.mode == "pnmix":
                b, h = divmod(u, self.Hkv)
                self.k_groups[u].append(quantize_k_h3l1_group(kg, self.high[b, h]))
            else:
                S = sensitivity(kg, self.sal_bits)
                A = salience(np.asarray(imp, np.float32), S)
                if self.tier_mode == "rank":
                    tiers = tiers_rank(A, self.n_bf16, self.n_uint4)
                else:
                    tiers = tiers_capped(A, self.tau_bf16, self.tau_uint4, self.n_bf16,
                                         self.n_uint4)
                self.k_groups[u].append(quantize_k_mixed_group(kg, tiers))
        self.v_parts[u].append(quantize_v_unit(vb, self.Gv, self.v_bits))

    # ------------------------------------------------------------- readers
    def dequant_unit(self, u: int):
        """fp64 K^, V^: the sink (exact), the quantized history, the residual."""
        D = self.D
        ks = []
        for grp in self.k_groups[u]:
            if self.mode == "uniform":
                ks.append(dequant_k_unit(*grp, self.Gk, self.k_bits))
            elif self.mode == "pnmix":
                codes, off, sc = grp
                ks.append(off.astype(np.float64)[None, :] +
                          sc.astype(np.float64)[None, :] * codes.astype(np.float64))
            else:
                ks.append(dequant_k_mixed_group(grp, self.Gk))
        vs = [dequant_v_unit(*part, self.Gv, self.v_bits) for part in self.v_parts[u]]
        kq = np.concatenate(ks) if ks else np.zeros((0, D))
        vq = np.concatenate(vs) if vs else np.zeros((0, D))
        kr = bf16_to_f32(self.res_k[u, :self.r]).astype(np.float64)
        vr = bf16_to_f32(self.res_v[u, :self.r]).astype(np.float64)
        ks = bf16_to_f32(self.sink_k[u, :self.s]).astype(np.float64)
        vs = bf16_to_f32(self.sink_v[u, :self.s]).astype(np.float64)
        return np.concatenate([ks, kq, kr]), np.concatenate([vs, vq, vr])

    def attention(self, q: np.ndarray, units=None) -> np.ndarray:
        """q bf16 bits [B, Hq, D] -> fp64 [B, Hq, D] (rows of units not in
        ``units`` are left NaN).  Query head h reads KV head h // n_rep."""
        B, Hq, D = q.shape
        n_rep = Hq // self.Hkv
        if self.s + self.T_q + self.r == 0:
            raise ValueError("attention over an empty cache")
        out = np.full((B, Hq, D), np.nan)
        qf = bf16_to_f32(q).astype(np.float64)
        for u in (range(B * self.Hkv) if units is None else units):
            b, h = divmod(u, self.Hkv)
            K, V = self.dequant_unit(u)
            for i in range(n_rep):
                out[b, h * n_rep + i] = attention(qf[b, h * n_rep + i], K, V)
        return out

    def export_uniform(self, u: int):
        """Canonical arrays of one unit: K codes/kmin/kscale over all groups,
        V codes/vmin/vscale over all quantized tokens."""
        kc = np.concatenate([g[0] for g in self.k_groups[u]]) if self.k_groups[u] else None
        km = np.concatenate([g[1] for g in self.k_groups[u]]) if self.k_groups[u] else None
        ks = np.concatenate([g[2] for g in self.k_groups[u]]) if self.k_groups[u] else None
        vc = np.concatenate([p[0] for p in self.v_parts[u]]) if self.v_parts[u] else None
        vm = np.concatenate([p[1] for p in self.v_parts[u]]) if self.v_parts[u] else None
        vs = np.concatenate([p[2] for p in self.v_parts[u]]) if self.v_parts[u] else None
        return kc, km, ks, vc, vm, vs


class KiviOracleCache:
    """KIVI's streaming cache ("KIVI: KV cache axes" §4–§6), in its
    Algorithm 1 order (append, then adjust both caches, then attend), for
    B x Hkv units of head dimension D:

    - Key: a new token joins the key residual; when it holds R tokens they
      are quantized per channel in groups of G tokens and the residual
      empties, so 0 <= r_K < R after every step.
    - Value: a FIFO; a new token joins the value residual, and when it holds
      more than R tokens the oldest leaves it, quantized per token in groups
      of G channels, so r_V = min(tokens, R).
    - Origins and steps in bf16, computed in bf16 (§7; quantize_group_bf16).
    - Attention: one softmax over all visible tokens in order; the value
      rows follow the value boundary, not the key boundary (§6).

    Prefill of L tokens leaves the state L appends would (the persisted
    invariants of §5): L - L mod R keys quantized, the last min(L, R)
    values in the FIFO.
    """

    def __init__(self, B, Hkv, D, k_bits=2, v_bits=2, G=32, R=128):
        if R % G or D % G:
            raise ValueError("R and D must be multiples of G")
        self.B, self.Hkv, self.D = B, Hkv, D
        self.k_bits, self.v_bits, self.G, self.R = k_bits, v_bits, G, R
        U = B * Hkv
        self.kq = [[] for _ in range(U)]   # per G-token group: codes [G][D], origin [D], step [D]
        self.vq = [[] for _ in range(U)]   # per token: codes [D], origin [D/G], step [D/G]
        self.kr = [[] for _ in range(U)]   # bf16 bit rows [D]
        self.vr = [[] for _ in range(U)]

    def _seal_keys(self, u):
        rows = np.stack(self.kr[u]).astype(np.uint16)          # [R][D]
        x = bf16_to_f32(rows)
        for g0 in range(0, self.R, self.G):
            codes = np.zeros((self.G, self.D), np.uint8)
            origin = np.zeros(self.D, np.uint16)
            step = np.zeros(self.D, np.uint16)
            for d in range(self.D):
                codes[:, d], origin[d], step[d] = quantize_group_bf16(x[g0:g0 + self.G, d],
                                                                      self.k_bits)
            self.kq[u].append((codes, origin, step))
        self.kr[u] = []

    def _seal_value(self, u):
        row = bf16_to_f32(np.asarray(self.vr[u].pop(0), np.uint16))
        nj = self.D // self.G
        codes = np.zeros(self.D, np.uint8)
        origin = np.zeros(nj, np.uint16)
        step = np.zeros(nj, np.uint16)
        for j in range(nj):
            sl = slice(j * self.G, (j + 1) * self.G)
            codes[sl], origin[j], step[j] = quantize_group_bf16(row[sl], self.v_bits)
        self.vq[u].append((codes, origin, step))

    def append(self, k_new: np.ndarray, v_new: np.ndarray):
        """One token, bf16 bits [B, Hkv, D] each."""
        k_new = np.asarray(k_new, np.uint16).reshape(-1, self.D)
        v_new = np.asarray(v_new, np.uint16).reshape(-1, self.D)
        for u in range(self.B * self.Hkv):
            self.kr[u].append(k_new[u].copy())
            if len(self.kr[u]) == self.R:
                self._seal_keys(u)
            self.vr[u].append(v_new[u].copy())
            if len(self.vr[u]) > self.R:
                self._seal_value(u)

    def prefill(self, K: np.ndarray, V: np.ndarray):
        """K, V bf16 bits [B, Hkv, L, D] into an empty cache."""
        if any(self.kq[u] or self.kr[u] or self.vq[u] or self.vr[u]
               for u in range(self.B * self.Hkv)):
            raise ValueError("prefill into a non-empty cache")
        B, Hkv, L, D = K.shape
        n_k = L - L % self.R
        n_v = L - min(L, self.R)
        for u in range(B * Hkv):
            b, h = divmod(u, Hkv)
            for t0 in range(0, n_k, self.R):
                self.kr[u] = [K[b, h, t] for t in range(t0, t0 + self.R)]
                self._seal_keys(u)
            self.kr[u] = [K[b, h, t] for t in range(n_k, L)]
            self.vr[u] = [V[b, h, t] for t in range(L)]
            for _ in range(n_v):
                self._seal_value(u)

    def lengths(self, u: int = 0):
        """(quantized keys, key residual, quantized values, value residual)."""
        return (self.G * len(self.kq[u]), len(self.kr[u]), len(self.vq[u]), len(self.vr[u]))

    def dequant_unit(self, u: int):
        """fp64 K^, V^ of one unit, one row per visible token in order."""
        D, G = self.D, self.G
        ks = [bf16_to_f32(o).astype(np.float64)[None, :] +
              bf16_to_f32(s).astype(np.float64)[None, :] * c.astype(np.float64)
              for c, o, s in self.kq[u]]
        vs = []
        for c, o, s in self.vq[u]:
            vs.append(np.repeat(bf16_to_f32(o).astype(np.float64), G) +
                      np.repeat(bf16_to_f32(s).astype(np.float64), G) * c.astype(np.float64))
        kq = np.concatenate(ks) if ks else np.zeros((0, D))
        vq = np.stack(vs) if vs else np.zeros((0, D))
        kr = (bf16_to_f32(np.stack(self.kr[u]).astype(np.uint16)).astype(np.float64)
              if self.kr[u] else np.zeros((0, D)))
        vr = (bf16_to_f32(np.stack(self.vr[u]).astype(np.uint16)).astype(np.float64)
              if self.vr[u] else np.zeros((0, D)))
        return np.concatenate([kq, kr]), np.concatenate([vq, vr])

    def attention(self, q: np.ndarray) -> np.ndarray:
        """q bf16 bits [B, Hq, D] -> fp64 [B, Hq, D]; query head h reads KV
        head h // n_rep."""
        B, Hq, D = q.shape
        n_rep = Hq // self.Hkv
        out = np.zeros((B, Hq, D))
        qf = bf16_to_f32(q).astype(np.float64)
        for u in range(B * self.Hkv):
            b, h = divmod(u, self.Hkv)
            K, V = self.dequant_unit(u)
            if K.shape[0] == 0:
                raise ValueError("attention over an empty cache")
            for i in range(n_rep):
                out[b, h * n_rep + i] = attention(qf[b, h * n_rep + i], K, V)
        return out
