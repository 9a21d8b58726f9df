"""Shared helpers for the GPU parity tests: run the same seeded inputs
through libkvq (via the binding) and through the CPU oracle, and compare.

Acceptance (stated once, used everywhere):
  - codes, origins (bf16) and steps (fp32): bit-exact;
  - tiers and channel permutations: exact;
  - attention output, per (batch, query head) row:
      ||o_gpu - o_ref||_2 <= 2e-3 * ||o_ref||_2   and
      max|o_gpu - o_ref|  <= 5e-3 * max|o_ref|,
    o_ref the oracle's fp64 attention over its own dequantized cache.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
import bit_kv_cache_kvq_gb300 as kvq
from bit_kv_cache_kvq_gb300.workloads import bf16_bits

REL_L2 = 2e-3
MAX_ABS_FRAC = 5e-3


def assert_attention_close(gpu_out: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = gpu_out.detach().double().cpu().numpy().reshape(-1, ref.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    checked = 0
    for i in range(r.shape[0]):
        if np.isnan(r[i, 0]):
            continue
        err = g[i] - r[i]
        nr = np.linalg.norm(r[i])
        assert np.all(np.isfinite(g[i])), f"{what} row {i}: non-finite output"
        assert np.linalg.norm(err) <= REL_L2 * nr, \
            f"{what} row {i}: rel L2 {np.linalg.norm(err) / nr:.3e}"
        assert np.max(np.abs(err)) <= MAX_ABS_FRAC * np.max(np.abs(r[i])), \
            f"{what} row {i}: max abs {np.max(np.abs(err)):.3e} vs {np.max(np.abs(r[i])):.3e}"
        checked += 1
    assert checked > 0
    return checked


def f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


class UnitOracles:
    """One oracle cache per sampled (b, kv head) unit, fed the same bf16
    inputs as the GPU cache."""

    def __init__(self, units, Hkv, k_bits=2, v_bits=2, mode="uniform", n_bf16=0, n_uint4=0,
                 n_sink=0, tier_mode="rank", tau_bf16=0.0, tau_uint4=0.0):
        self.units = list(units)
        self.Hkv = Hkv
        self.caches = [orc.OracleCache(1, 1, 128, k_bits, v_bits, mode=mode, n_bf16=n_bf16,
                                       n_uint4=n_uint4, n_sink=n_sink, tier_mode=tier_mode,
                                       tau_bf16=tau_bf16, tau_uint4=tau_uint4)
                       for _ in self.units]

    def _sel(self, t: torch.Tensor, u: int):
        b, h = divmod(u, self.Hkv)
        return bf16_bits(t[b:b + 1, h:h + 1])

    def prefill(self, K, V, importance=None):
        for u, c in zip(self.units, self.caches):
            b, h = divmod(u, self.Hkv)
            imp = None if importance is None else importance[b:b + 1, h:h + 1].cpu().numpy()
            c.prefill(self._sel(K, u), self._sel(V, u), imp)

    def append(self, k_new, v_new):
        for u, c in zip(self.units, self.caches):
            b, h = divmod(u, self.Hkv)
            c.append(bf16_bits(k_new[b:b + 1, h:h + 1]), bf16_bits(v_new[b:b + 1, h:h + 1]))

    def observe(self, q: torch.Tensor):
        n_rep = q.shape[1] // self.Hkv
        for u, c in zip(self.units, self.caches):
            b, h = divmod(u, self.Hkv)
            c.observe(bf16_bits(q[b:b + 1, h * n_rep:(h + 1) * n_rep]))

    def flush(self, importance=None):
        for u, c in zip(self.units, self.caches):
            b, h = divmod(u, self.Hkv)
            c.flush(None if importance is None else importance[b:b + 1, h:h + 1].cpu().numpy())

    def attention(self, q: torch.Tensor) -> np.ndarray:
        """fp64 [B, Hq, D] with NaN rows for units not sampled."""
        B, Hq, D = q.shape
        n_rep = Hq // self.Hkv
        out = np.full((B, Hq, D), np.nan)
        for u, c in zip(self.units, self.caches):
            b, h = divmod(u, self.Hkv)
            qs = bf16_bits(q[b:b + 1, h * n_rep:(h + 1) * n_rep])
            out[b, h * n_rep:(h + 1) * n_rep] = c.attention(qs)[0]
        return out


def assert_uniform_exports_equal(cache: kvq.KVCache, ref: UnitOracles):
    kc, km, ks = cache.export_k()
    vc, vm, vs = cache.export_v()
    kr, vr = cache.export_residual()
    torch.cuda.synchronize()
    kc, km, ks = kc.cpu().numpy(), bf16_bits(km), f32_bits(ks)
    vc, vm, vs = vc.cpu().numpy(), bf16_bits(vm), f32_bits(vs)
    krb, vrb = bf16_bits(kr), bf16_bits(vr)
    for u, oc in zip(ref.units, ref.caches):
        b, h = divmod(u, ref.Hkv)
        okc, okm, oks, ovc, ovm, ovs = oc.export_uniform(0)
        if okc is None:
            assert kc.shape[2] == 0 and vc.shape[2] == 0
        else:
            assert np.array_equal(kc[b, h], okc), f"K codes differ (unit {u})"
            assert np.array_equal(km[b, h], okm), f"K origins differ (unit {u})"
            assert np.array_equal(ks[b, h], oks.view(np.uint32)), f"K steps differ (unit {u})"
            assert np.array_equal(vc[b, h], ovc), f"V codes differ (unit {u})"
            assert np.array_equal(vm[b, h], ovm), f"V origins differ (unit {u})"
            assert np.array_equal(vs[b, h], ovs.view(np.uint32)), f"V steps differ (unit {u})"
        r = oc.r
        assert np.array_equal(krb[b, h], oc.res_k[0, :r]), f"K residual differs (unit {u})"
        assert np.array_equal(vrb[b, h], oc.res_v[0, :r]), f"V residual differs (unit {u})"


def assert_mixed_exports_equal(cache: kvq.KVCache, ref: UnitOracles):
    """Mixed keys: permutation, raw BF16 tier, UINT4/UINT2 codes, origins and
    steps per group; values and residual as in the uniform case."""
    t = cache.export_k_mixed()
    counts = t["counts"].cpu().numpy()
    vc, vm, vs = cache.export_v()
    kr, vr = cache.export_residual()
    torch.cuda.synchronize()
    perm, c4, c2 = t["perm"].cpu().numpy(), t["c4"].cpu().numpy(), t["c2"].cpu().numpy()
    raw, m4, m2 = bf16_bits(t["raw"]), bf16_bits(t["m4"]), bf16_bits(t["m2"])
    s4, s2 = f32_bits(t["s4"]), f32_bits(t["s2"])
    vc, vm, vs = vc.cpu().numpy(), bf16_bits(vm), f32_bits(vs)
    krb, vrb = bf16_bits(kr), bf16_bits(vr)
    for u, oc in zip(ref.units, ref.caches):
        b, h = divmod(u, ref.Hkv)
        groups = oc.k_groups[0]
        assert perm.shape[2] == len(groups)
        for gi, grp in enumerate(groups):
            where = f"(unit {u}, group {gi})"
            nb, n4, n2 = grp.raw.shape[0], grp.c4.shape[0], grp.c2.shape[0]
            assert tuple(counts[b, h, gi]) == (nb, n4), f"tier counts differ {where}"
            assert np.array_equal(perm[b, h, gi], grp.perm), f"permutation differs {where}"
            # the export has the record's room per tier; rows past the group's
            # own count are zero
            for name, got, want in (("BF16 tier", raw, grp.raw), ("UINT4 codes", c4, grp.c4),
                                    ("UINT4 origins", m4, grp.m4),
                                    ("UINT4 steps", s4, grp.s4.view(np.uint32)),
                                    ("UINT2 codes", c2, grp.c2), ("UINT2 origins", m2, grp.m2),
                                    ("UINT2 steps", s2, grp.s2.view(np.uint32))):
                g = got[b, h, gi]
                n = want.shape[0]
                assert np.array_equal(g[:n], want), f"{name} differ {where}"
                assert not g[n:].any(), f"{name} padding not zero {where}"
        parts = oc.v_parts[0]
        if parts:
            ovc, ovm, ovs = (np.concatenate([p[i] for p in parts]) for i in range(3))
            assert np.array_equal(vc[b, h], ovc), f"V codes differ (unit {u})"
            assert np.array_equal(vm[b, h], ovm), f"V origins differ (unit {u})"
            assert np.array_equal(vs[b, h], ovs.view(np.uint32)), f"V steps differ (unit {u})"
        r = oc.r
        assert np.array_equal(krb[b, h], oc.res_k[0, :r]), f"K residual differs (unit {u})"
        assert np.array_equal(vrb[b, h], oc.res_v[0, :r]), f"V residual differs (unit {u})"


def assert_sink_equal(cache: kvq.KVCache, ref: UnitOracles):
    """The attention-sink window, bit-exact, and its length."""
    ks, vs = cache.export_sink()
    torch.cuda.synchronize()
    ksb, vsb = bf16_bits(ks), bf16_bits(vs)
    for u, oc in zip(ref.units, ref.caches):
        b, h = divmod(u, ref.Hkv)
        assert cache.sink_tokens() == oc.s
        assert np.array_equal(ksb[b, h], oc.sink_k[0, :oc.s]), f"K sink differs (unit {u})"
        assert np.array_equal(vsb[b, h], oc.sink_v[0, :oc.s]), f"V sink differs (unit {u})"
