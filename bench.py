#!/usr/bin/env python3
"""Quantized-KV decode benchmark (one JSON line on rank 0).

Workload (default): Llama-3.1-8B-shaped GQA decode layer, 32 query / 8 KV
heads, D = 128, batch 16, 32768 quantized tokens + 100 residual tokens, K and
V at 2 bits (K per channel over 128-token groups, V per token over 32
channels), synthetic seeded bf16 inputs with 4 outlier key channels per KV
head.

A step is one MixKVQ Algorithm 1 decode step through the C ABI
(kvq_decode_step): append the new token's key/value to the residual, flush
(quantize 128 tokens) when the residual is full, then the fused split-K
decode attention (partial + combine); without a flush the decode kernel
writes the token itself, so a step is the decode launch and its combine.  The quantized history starts below the workload's length by half
the groups the timed steps will flush, so the mean context over the timed
region is the workload's.

metric/value: effective HBM GB/s = algorithmic bytes of the steps (packed
cache 94 B/token/KV head at 2 bits, residual 512 B/token, q and o, append and
flush traffic) / device time of the K steps between two events.  The
roofline object covers the dominant kernel, the split-K decode kernel: its
mean launch duration over 50 calls, each from an event recorded before the
call to the event the library records between the decode kernel and its
combine (kvq_set_decode_split_event); 50 more calls, interleaved, between
two events give the whole call (decode + combine) as p10/p50/p90.  Every
call runs after a scratch write of twice the L2 size (then a read of another
buffer as large, so no dirty line is written back during the call) outside
the events.  e2e repeats the steps through the same API with q, k_new
and v_new copied from pinned host memory (one packed copy) and the output
copied back every step, the host reading each output one step later.
cpu_baseline times the CPU oracle on a bounded sample.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attention: effective HBM GB/s (% of peak), µs/step"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024      # GB300 L2
ATTN_REPS = 50                     # timed calls of each kind (kernel alone / whole call)

# dram__bytes_read.sum + dram__bytes_write.sum of one decode_mma_kernel
# launch over its algorithmic bytes, from the ncu captures kept under
# profiles/, keyed by the hash of the decode kernel's code they were taken
# on (a stale entry reports null); the bench reports that ratio times the
# timed launches' mean algorithmic bytes (traffic per unit does not depend
# on the batch, and the captured step's context is the workload's).
# Llama-8B, captured at batch 8 (64 units, 32768 + 100 tokens, the token
# append fused): 200.988 MB read + 3.793 MB written against 200.638 MB
# (mostly the split-K partials written).  MixKVQ, captured at the bench size
# (batch 8, 16384 + 100 tokens): 124.507 MB read + 2.954 MB written against
# 120.64 MB (the stored mixed key records are 7552 B against 7100 B of
# algorithmic key bytes per group).
NCU_TRAFFIC = {
    "65b84ef42b3a8a09": {
        ("llama8b_gqa_32k_b16", 16, 32768, 2): 204.780544 / 200.638464,
        ("mixkvq_qwen32b_16k_b8", 8, 16384, 2): 127.460864 / 120.64,
    },
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1024)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama8b_gqa_32k_b16")
    p.add_argument("--batch", type=int, default=0, help="override the batch (profiling)")
    p.add_argument("--context", type=int, default=0, help="override quantized tokens")
    p.add_argument("--bits", type=int, default=0, help="override k/v bits")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-bf16", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--sweep", action="store_true",
                   help="long-context sweep: one JSON line per context x batch x bits point "
                        "(decode steps and the bf16 comparator; no e2e or CPU legs)")
    return p.parse_args()


# --------------------------------------------------------------- clocks
class ClockSampler(threading.Thread):
    """Samples SM clock and clock-event reasons through NVML while running."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, period_s=0.002):
        super().__init__(daemon=True)
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._halt = threading.Event()
        self.ok = False
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            import torch
            idx = torch.cuda.current_device()
            ids = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
            if idx < len(ids) and ids[idx].isdigit():
                idx = int(ids[idx])             # NVML counts physical devices
            if self.nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def run(self):
        if not self.ok:
            return
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        getr = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._halt.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if getr(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.period)

    def stop(self):
        self._halt.set()
        self.join(timeout=1.0)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples),
                "reasons": [n for b, n in self.REASONS.items() if self.reasons & b]}


def percentiles(xs, ps):
    """Nearest-rank percentiles of a list."""
    ys = sorted(xs)
    return [ys[min(len(ys) - 1, max(0, int(round(p / 100 * (len(ys) - 1)))))] for p in ps]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """sha256 of the decode kernel's sources with // comments and blank
    space dropped, so the key follows the code, not its comments."""
    import re
    h = hashlib.sha256()
    for name in ("decode_mma.cuh", "decode_mma.cu", "frag_layout.h", "kvq_internal.h", "mma_util.h"):
        with open(os.path.join(ROOT, "bit_kv_cache_kvq_gb300", "csrc", name)) as f:
            for line in f:
                code = re.sub(r"//.*", "", line).strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


# ------------------------------------------------------ algorithmic bytes
def mixed_k_group_bytes(w):
    """Mixed key group: permutation, raw BF16 tier, UINT4 and UINT2 codes and
    an (fp32 step, bf16 origin) per quantized channel (7100 B at 6/25/97)."""
    n2 = 128 - w.n_bf16 - w.n_uint4
    return 128 + w.n_bf16 * 256 + w.n_uint4 * 64 + n2 * 32 + (w.n_uint4 + n2) * 6


def kivi_half_bytes(w):
    """KIVI variant, one token's key (or value): codes plus a bf16 origin and
    step per 32-element group (the KIVI article's 3 bits per element at 2 bits)."""
    return 128 * w.k_bits // 8 + 16


def pnmix_k_bytes(w):
    """PN-Mix key bytes per token: the LSB plane (1 bit a channel), the upper
    two bits of the 2 n_high_pairs high channels, an fp32 offset and scale
    per channel and 128-token group."""
    nh = 2 * w.extra.get("n_high_pairs", 32)
    return 128 / 8 + nh * 2 / 8 + 128 * 8 / 128


def token_bytes(w):
    """Algorithmic bytes of one quantized token of one (b, kv head)."""
    if w.mode == "kivi":
        return 2 * kivi_half_bytes(w)
    if w.mode == "pnmix":
        return pnmix_k_bytes(w) + 128 * w.v_bits // 8 + 24
    v = 128 * w.v_bits // 8 + 24
    if w.mode == "mixed":
        return mixed_k_group_bytes(w) / 128 + v
    return 128 * w.k_bits // 8 + 6 + v


def attention_bytes(w, T_q, r):
    """Packed cache + bf16 residual + q (bf16) + o (fp32) of one decode
    attention call.  KIVI: T_q quantized keys and r bf16 residual keys; of the
    T_q + r values the last min(T_q + r, 128) are bf16 (the FIFO)."""
    U = w.B * w.Hkv
    qo = w.B * w.Hq * (256 + 512)
    if w.mode == "kivi":
        fifo = min(T_q + r, 128)
        return U * ((T_q + T_q + r - fifo) * kivi_half_bytes(w) + (r + fifo) * 256) + qo
    return U * (T_q * token_bytes(w) + r * 512) + qo


def append_bytes(w):
    """Read k_new, v_new; write the residual slots (KIVI: and the value
    leaving the FIFO, read and written quantized)."""
    extra = 256 + kivi_half_bytes(w) if w.mode == "kivi" else 0
    return w.B * w.Hkv * (2 * 2 * 256 + extra)


def flush_bytes(w):
    return w.B * w.Hkv * 128 * (512 + token_bytes(w))


# ------------------------------------------------------------- multi-rank
def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the slowest rank's time); x itself
    for one rank.  Ranks shard whole (batch row, KV head) units, so this
    and a barrier are the only cross-rank traffic."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_workload(w, rank: int):
    """Weak scaling: every rank decodes its own batch of the workload (its
    own (batch row, KV head) units), drawn from seeds offset by the rank."""
    from bit_kv_cache_kvq_gb300.workloads import scaled
    return scaled(w, seed=w.seed + 100 * rank)


# ---------------------------------------------------------------- arms
def workload_from(args):
    from bit_kv_cache_kvq_gb300.workloads import WORKLOADS, scaled, sweep_workload
    if args.workload.startswith("sweep_c"):      # sweep_c<context>_b<batch>_k<bits>
        c, b, k = (int(x[1:]) for x in args.workload[len("sweep_"):].split("_"))
        w = sweep_workload(c, b, k)
    else:
        w = WORKLOADS[args.workload]
    ch = {}
    if args.batch:
        ch["B"] = args.batch
    if args.context:
        ch["T_q"] = args.context
    if args.bits:
        ch["k_bits"] = ch["v_bits"] = args.bits
    return scaled(w, **ch) if ch else w


def config_of(w, extra=None):
    c = {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": 128,
         "quantized_tokens": w.T_q, "residual_tokens": w.r, "k_bits": w.k_bits,
         "v_bits": w.v_bits, "k_group_tokens": 128, "v_group_channels": 32}
    if w.mode == "mixed":
        c.update({"k_mode": "mixed", "n_bf16": w.n_bf16, "n_uint4": w.n_uint4,
                  "n_uint2": 128 - w.n_bf16 - w.n_uint4, "query_window": w.Lq})
    if w.mode == "kivi":
        c.update({"k_mode": "kivi", "k_group_tokens": 32, "key_seal_tokens": 128,
                  "value_fifo_tokens": 128, "metadata": "bf16"})
    if w.mode == "pnmix":
        c.update({"k_mode": "pnmix", "n_high_pairs": w.extra.get("n_high_pairs", 32),
                  "high_bits": 3, "low_bits": 1, "pair_layout": "adjacent",
                  "query_window": w.Lq})
    if extra:
        c.update(extra)
    return c


class OracleSample:
    """A few (batch row, KV head) units of the workload, quantized by the CPU
    oracle (untimed); time_step() times the oracle's decode attention
    (dequantize + fp64 attention of the unit's n_rep query heads) on one."""

    def __init__(self, w, n_units):
        import oracle as orc
        from bit_kv_cache_kvq_gb300.workloads import (bf16_bits, make_kv, make_q,
                                                      make_query_window, scaled)
        oracle_mod = orc
        self.one = scaled(w, B=1, Hkv=1, Hq=w.n_rep, k_outliers=min(w.k_outliers, 4))
        self.units = []
        for j in range(n_units):
            u = scaled(self.one, seed=self.one.seed + 17 * j)
            K, V = make_kv(u)
            if u.mode == "pnmix":
                qw = bf16_bits(make_query_window(u)[0])
                sig = orc.pair_scores(qw, bf16_bits(K[0, 0]), orc.PAIR_ADJACENT)
                high = orc.channel_mask(orc.select_pairs(sig, u.extra.get("n_high_pairs", 32)),
                                        orc.PAIR_ADJACENT)[None, None]
                c = oracle_mod.OracleCache(1, 1, 128, u.k_bits, u.v_bits, mode="pnmix",
                                           high_channels=high)
                c.prefill(bf16_bits(K), bf16_bits(V))
                self.units.append((u, c, [bf16_bits(make_q(u, step=s)) for s in range(4)]))
                continue
            if u.mode == "kivi":
                c = oracle_mod.KiviOracleCache(1, 1, 128, u.k_bits, u.v_bits)
                c.prefill(bf16_bits(K), bf16_bits(V))
                c.T_q, c.r = c.lengths()[:2]
                self.units.append((u, c, [bf16_bits(make_q(u, step=s)) for s in range(4)]))
                continue
            c = oracle_mod.OracleCache(1, 1, 128, u.k_bits, u.v_bits, mode=u.mode,
                                       n_bf16=u.n_bf16, n_uint4=u.n_uint4)
            imp = None
            if u.mode == "mixed":
                imp = orc.importance(bf16_bits(make_query_window(u)[0]))[None, None]
            c.prefill(bf16_bits(K), bf16_bits(V), imp)
            self.units.append((u, c, [bf16_bits(make_q(u, step=s)) for s in range(4)]))
        self.calls = 0

    def time_step(self):
        import numpy as np
        u, c, qs = self.units[self.calls % len(self.units)]
        q = qs[(self.calls // len(self.units)) % len(qs)]
        self.calls += 1
        t0 = time.perf_counter()
        out = c.attention(q)
        sec = time.perf_counter() - t0
        assert np.all(np.isfinite(out))
        return attention_bytes(u, c.T_q, c.r), sec


def oracle_sample(w, seconds):
    """(bytes, seconds, calls) of the oracle over about `seconds` of work."""
    smp = OracleSample(w, 2)
    nbytes, spent = 0, 0.0
    while smp.calls == 0 or spent < seconds:
        nb, sec = smp.time_step()
        nbytes += nb
        spent += sec
    return nbytes, spent, smp.calls


def run_reference(args, rank, world):
    w = workload_from(args)
    if rank != 0:
        return None
    import oracle
    oracle.build()
    smp = OracleSample(w, 2)
    nbytes_tot, secs_tot = 0, 0.0
    for i in range(args.warmup + args.steps):
        nb, sec = smp.time_step()
        if i >= args.warmup:
            nbytes_tot += nb
            secs_tot += sec
    gbs = nbytes_tot / secs_tot / 1e9
    sample = (f"per step: one (batch row, KV head) unit, its {w.n_rep} query heads over "
              f"{w.T_q} quantized + {w.r} residual tokens (dequantize + fp64 attention)")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs_tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


def run_ours(args, rank, world):
    import torch
    import bit_kv_cache_kvq_gb300 as kvq
    from bit_kv_cache_kvq_gb300 import _build
    from bit_kv_cache_kvq_gb300.workloads import (make_kv, make_q, make_query_window,
                                                  make_token, scaled)

    _build.build()
    kvq.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    w0 = workload_from(args)
    w = rank_workload(w0, rank)                    # weak scaling: each rank its own batch
    K, W = args.steps, args.warmup
    n_flush = (w.r + K) // 128                     # flushes inside the timed steps
    T0 = max(0, w.T_q - 128 * (n_flush // 2))     # mean context over the timed steps ~ workload's
    L0 = T0 + w.r - W                              # prefill; the warm-up appends reach T0 + r
    if L0 < 0:
        raise SystemExit("--warmup exceeds the workload's tokens")
    cap = T0 + 128 * (n_flush + 2)

    Kall, Vall = make_kv(w, L=w.T_q + w.r, device=dev)
    toks = [make_token(w, i, device=dev) for i in range(W + K)]
    n_q = min(W + K, 64)
    qs = [make_q(w, step=i, device=dev) for i in range(n_q)]
    importance = None
    if w.mode == "mixed":   # MixKVQ: I_d from the query window, on the GPU
        importance, _, _ = kvq.channel_saliency(make_query_window(w, device=dev),
                                                Kall[:, :, :128].contiguous(), 2,
                                                n_bf16=w.n_bf16, n_uint4=w.n_uint4)
    cache = kvq.KVCache(w.B, w.Hkv, cap, w.k_bits, w.v_bits, mode=w.mode, n_bf16=w.n_bf16,
                        n_uint4=w.n_uint4, device=dev,
                        n_high_pairs=w.extra.get("n_high_pairs", 0))
    qwin = make_query_window(w, device=dev) if w.mode == "pnmix" else None
    out = torch.empty(w.B, w.Hq, 128, dtype=torch.float32, device=dev)
    ws = cache.workspace(w.Hq)
    stream = torch.cuda.current_stream()
    K0, V0 = Kall[:, :, :L0].contiguous(), Vall[:, :, :L0].contiguous()

    def prefill():
        cache.reset()
        if qwin is not None:     # PN-Mix: Eq. 6 pair selection, once per prefill
            cache.pnmix_pairs(qwin, K0)
        cache.prefill(K0, V0, importance=importance)

    # prefill quantize (kvq_quantize_prefill) on its own: bf16 K, V read once,
    # packed groups written, the L mod 128 tail copied to the residual
    for _ in range(2):
        prefill()
    pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p_reps = 5
    pa.record(stream)
    for _ in range(p_reps):
        prefill()
    pb.record(stream)
    torch.cuda.synchronize()
    prefill_us = 1e3 * pa.elapsed_time(pb) / p_reps
    n_grp = L0 // 128
    prefill_nb = w.B * w.Hkv * (L0 * 512 + n_grp * 128 * token_bytes(w) + (L0 % 128) * 512)

    def step(i, ev=None):
        """One decode step (kvq_decode_step: append, flush when the residual
        fills, attention); returns (launches, algorithmic bytes, bytes of the
        call).  Without a flush the decode kernel does the append itself."""
        kn, vn = toks[i]
        flushes = cache.lengths()[1] + 1 == 128
        if ev is not None:
            ev[0].record(stream)
        cache.decode_step(kn, vn, qs[i % n_q], out=out, workspace=ws, importance=importance)
        if ev is not None:
            ev[1].record(stream)
        tq, r = cache.lengths()
        nb = append_bytes(w) + attention_bytes(w, tq, r) + (flush_bytes(w) if flushes else 0)
        return (4 if flushes else 2), nb, nb

    def warm():
        prefill()
        for i in range(W):
            step(i)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()

    # pass 1: the K steps bracketed by two events only (value, ms_per_step)
    warm()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler()
    clk.start()
    time.sleep(0.02)
    # a ~0.5 ms busy kernel before the first event, so the host has queued
    # the first steps when the timed region starts (the device never waits
    # on the host's first submissions inside it)
    torch.cuda._sleep(1_000_000)
    t_start.record(stream)
    launches = 0
    total_bytes = 0
    for i in range(K):
        n, nb, _ = step(W + i)
        launches += n
        total_bytes += nb
    t_end.record(stream)
    torch.cuda.synchronize()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    # pass 2 (roofline): 2 x ATTN_REPS decode attention calls (kvq_decode_step:
    # the decode with the token append fused, and its combine), with a
    # scratch buffer twice the L2 size written before every call outside the
    # events.  Even calls run between two events on the launching stream (the
    # call's time); odd calls also have the library record an event between
    # the decode kernel and its combine (kvq_set_decode_split_event), so the
    # first event and that one bracket the decode kernel alone (the roofline
    # kernel's launch duration).  The residual starts ATTN_REPS tokens below
    # the workload's, so the calls never flush and their mean context is the
    # workload's.
    R, Wp = ATTN_REPS, 3
    R2 = 2 * R
    r0 = max(0, w.r - R2 // 2 - Wp)
    if r0 + Wp + R2 >= 128:
        r0 = 127 - Wp - R2
    Lp = w.T_q + r0
    Kp, Vp = Kall[:, :, :Lp].contiguous(), Vall[:, :, :Lp].contiguous()
    cache.reset()
    if qwin is not None:
        cache.pnmix_pairs(qwin, Kp)
    cache.prefill(Kp, Vp, importance=importance)
    del Kp, Vp
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sweep = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        """Write a buffer twice the L2 size, then read another as large: the
        timed call starts with none of its data in L2 and no dirty lines
        left to write back during it."""
        scratch.fill_(float(i))
        return sweep.sum()

    for i in range(Wp):                             # untimed warm-up calls
        kn, vn = toks[i % len(toks)]
        cache.decode_step(kn, vn, qs[i % n_q], out=out, workspace=ws, importance=importance)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(R2)]
    for ev in evs:
        ev[2].record(stream)                         # created before the timed calls
    attn_bytes = []
    for i in range(R2):
        flush_l2(i)                                  # outside the events
        tq_r = cache.lengths()
        kn, vn = toks[(Wp + i) % len(toks)]
        evs[i][0].record(stream)
        if i % 2:
            kvq.set_decode_split_event(evs[i][2])
        cache.decode_step(kn, vn, qs[i % n_q], out=out, workspace=ws, importance=importance)
        evs[i][1].record(stream)
        assert cache.lengths() == (tq_r[0], tq_r[1] + 1), "a timed call flushed"
        attn_bytes.append(append_bytes(w) + attention_bytes(w, tq_r[0], tq_r[1] + 1))
    torch.cuda.synchronize()
    clk.stop()
    del scratch, sweep
    if world > 1:
        torch.distributed.barrier()
    if args.no_e2e:
        del K0, V0
    if args.no_bf16 and args.no_e2e:       # keep device memory small (profiling)
        del Kall, Vall
        torch.cuda.empty_cache()
    attn_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(0, R2, 2)]
    kern_ms = [evs[i][0].elapsed_time(evs[i][2]) for i in range(1, R2, 2)]
    p10, p50, p90 = percentiles(attn_ms, (10, 50, 90))
    k10, k50, k90 = percentiles(kern_ms, (10, 50, 90))
    kern_mean = sum(kern_ms) / len(kern_ms)
    attn_avg_bytes = sum(attn_bytes) / R2
    kern_avg_bytes = sum(attn_bytes[1::2]) / R
    ms_per_step = elapsed_ms / K
    value = total_bytes * world / (elapsed_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    achieved = kern_avg_bytes / (kern_mean * 1e-3) / 1e9
    src_hash = kernel_source_hash()
    traffic_ratio = NCU_TRAFFIC.get(src_hash, {}).get((w.name, w.B, w.T_q, w.k_bits))
    traffic = None if traffic_ratio is None else traffic_ratio * kern_avg_bytes
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(w0, {
            "l2": "inputs larger than L2 (packed cache %.0f MB vs 129 MB L2)"
                  % (attention_bytes(w, w.T_q, w.r) / 1e6),
            "first_timed_context": T0 + w.r, "timed_flushes": n_flush,
            "per_rank_seed_offset": 100}),
        "us_per_step": 1e3 * ms_per_step,
        "decode_attention_us": 1e3 * p50,
        "decode_attention_us_p10_p50_p90": [1e3 * p10, 1e3 * p50, 1e3 * p90],
        "decode_kernel_us_mean": 1e3 * kern_mean,
        "decode_kernel_us_p10_p50_p90": [1e3 * k10, 1e3 * k50, 1e3 * k90],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": "decode_mma_kernel (split-K partials; the combine kernel "
                               "after it is in the call's time)",
                     "algorithmic_bytes_per_launch": kern_avg_bytes, "traffic": traffic,
                     "kernel_source": src_hash,
                     "call_frac": attn_avg_bytes / (p50 * 1e-3) / 1e9 / peak,
                     "timing": f"mean of {R} decode kernel launches, each from an event "
                               f"recorded before the call to one the library records between "
                               f"the decode kernel and its combine; call times (p10/p50/p90, "
                               f"call_frac from the median) from {R} calls between two events, "
                               f"interleaved; every call after a {2 * L2_BYTES / 1e6:.0f} MB "
                               f"scratch write (2x L2) and a read of another buffer as large, "
                               f"outside the events; residual {r0 + Wp + 1}..{r0 + Wp + R2} "
                               f"tokens"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "prefill": {"tokens": L0, "us": prefill_us,
                    "gbs": prefill_nb / (prefill_us * 1e-6) / 1e9,
                    "algorithmic_bytes": prefill_nb,
                    "note": "kvq_quantize_prefill alone, outside the timed decode steps"
                            + ("; includes the Eq. 6 pair selection" if w.mode == "pnmix" else "")},
    }

    # bf16 unquantized comparator at the same batch and context
    if not args.no_bf16:
        q0 = qs[0]
        for _ in range(3):
            kvq.decode_bf16(Kall, Vall, q0, out=out)
        nb16 = w.B * w.Hkv * (w.T_q + w.r) * 512 + w.B * w.Hq * (256 + 512)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record(stream)
        for _ in range(reps):
            kvq.decode_bf16(Kall, Vall, q0, out=out)
        b.record(stream)
        torch.cuda.synchronize()
        us16 = 1e3 * a.elapsed_time(b) / reps
        line["comparators"] = {"bf16_decode_us": us16,
                               "bf16_decode_gbs": nb16 / (us16 * 1e-6) / 1e9,
                               "bf16_bytes_per_step": nb16,
                               "speedup_vs_bf16": us16 / (1e3 * p50)}

    # e2e: host buffers, copies inside the timed region.  Every step copies
    # its inputs (k_new, v_new, q packed in one pinned buffer) to the device
    # in one copy and its output back to a pinned buffer.  The copies run on
    # a copy stream with two device staging buffers and two outputs, so step
    # i + 1's input copy and step i's output copy overlap the kernels; the
    # host reads step i's output after it has enqueued step i + 1.
    if not args.no_e2e:
        prefill()
        # at least 64 steps (a short host-timed loop is noisy), within the cache
        KE = max(1, min(max(K, 64), 256, cap - (L0 + W)))
        nk = toks[0][0].numel()
        h_in = []
        for i in range(W + KE + 1):
            kn, vn = toks[min(i, len(toks) - 1)]
            packed = torch.cat([kn.reshape(-1), vn.reshape(-1), qs[i % n_q].reshape(-1)])
            h_in.append(packed.cpu().pin_memory())
        d_in = [torch.empty_like(h_in[0], device=dev) for _ in range(2)]
        views = [(d[:nk].view(toks[0][0].shape), d[nk:2 * nk].view(toks[0][1].shape),
                  d[2 * nk:].view(qs[0].shape)) for d in d_in]
        outs = [torch.empty_like(out) for _ in range(2)]
        h_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        copy_s = torch.cuda.Stream(device=dev)
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "used", "out")}

        def h2d(i, j):      # inputs of step i into staging buffer j % 2
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(ev["used"][j % 2])   # step j - 2 is done with it
                d_in[j % 2].copy_(h_in[i], non_blocking=True)
                ev["in"][j % 2].record(copy_s)

        h_np = [h.numpy() for h in h_out]

        def step_bytes(n):
            """Algorithmic bytes of the next n steps from the cache's lengths
            now (host arithmetic: each step appends a token and flushes a
            full residual), so the timed loop makes no extra calls."""
            tq, r = cache.lengths()
            nbs = []
            for _ in range(n):
                flushes = r + 1 == 128
                tq, r = (tq + 128, 0) if flushes else (tq, r + 1)
                nbs.append(append_bytes(w) + (flush_bytes(w) if flushes else 0)
                           + attention_bytes(w, tq, r))
            return nbs, (tq, r)

        def compute(j):
            d_k, d_v, d_q = views[j % 2]
            stream.wait_event(ev["in"][j % 2])
            cache.decode_step(d_k, d_v, d_q, out=outs[j % 2], workspace=ws, importance=importance)
            ev["used"][j % 2].record(stream)
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(ev["used"][j % 2])
                h_out[j % 2].copy_(outs[j % 2], non_blocking=True)
                ev["out"][j % 2].record(copy_s)

        def consume(j):
            ev["out"][j % 2].synchronize()
            return float(h_np[j % 2][0, 0, 0])

        def run(first, n):
            acc = 0.0
            h2d(first, 0)
            for j in range(n):
                if j + 1 < n:
                    h2d(first + j + 1, j + 1)
                compute(j)
                if j >= 1:
                    acc += consume(j - 1)
            acc += consume(n - 1)
            return acc

        run(0, W)
        torch.cuda.synchronize()
        nbs, lengths_after = step_bytes(KE)
        e2e_bytes = sum(nbs)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        checksum = run(W, KE)
        t1 = time.perf_counter()
        assert cache.lengths() == lengths_after, "e2e step accounting"
        assert checksum == checksum, "e2e output is not finite"
        e2e_s = max_over_ranks(t1 - t0, world, dev)
        line["e2e"] = {"value": e2e_bytes * world / e2e_s / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": h_in[0].numel() * h_in[0].element_size(),
                       "d2h_bytes_per_step": out.numel() * 4,
                       "steps": KE, "us_per_step": 1e6 * e2e_s / KE,
                       "note": "one pinned H2D copy of k_new, v_new and q and one D2H copy "
                               "of the output per step, on a copy stream overlapping the "
                               "kernels; the host reads step i's output after enqueueing "
                               "step i+1"}

    # CPU oracle on a bounded sample (rank 0, N = 1 only)
    if not args.no_cpu and rank == 0 and world == 1:
        with one_core() as core:
            nb, sec, units = oracle_sample(w0, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": nb / sec / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{units} decode-attention calls, each one (batch row, KV head) unit "
                      f"of this workload with its {w0.n_rep} query heads over {w0.T_q} + "
                      f"{w0.r} tokens (dequantize + fp64 attention), {sec:.1f} s "
                      f"single-threaded, pinned to core {core}",
            "cpu_model": _cpu_model(), "host_cores": os.cpu_count()}
    return line


# Arm CPU part numbers (MIDR) of the hosts this runs on
_ARM_PARTS = {"0xd4f": "Arm Neoverse-V2 (NVIDIA Grace)", "0xd40": "Arm Neoverse-V1",
              "0xd0c": "Arm Neoverse-N1", "0xd49": "Arm Neoverse-N2"}


def _cpu_model():
    """A readable CPU model: lscpu's model name, else /proc/cpuinfo's model
    name, else the Arm part number mapped to its core name."""
    import platform
    import subprocess
    try:
        res = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in res.stdout.splitlines():
            if ln.strip().lower().startswith("model name"):
                name = ln.split(":", 1)[1].strip()
                if name and name != "-":
                    return name
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":", 1)[0].strip().lower()
                if key == "model name":
                    return ln.split(":", 1)[1].strip()
                if key == "cpu part":
                    part = ln.split(":", 1)[1].strip().lower()
                    return _ARM_PARTS.get(part, f"Arm part {part}") + f" ({platform.machine()})"
    except OSError:
        pass
    return platform.machine()


class one_core:
    """Pin the calling thread to one host core for the duration (the oracle is
    single-threaded); restores the previous affinity."""

    def __enter__(self):
        self.prev = None
        try:
            self.prev = os.sched_getaffinity(0)
            core = max(self.prev)
            os.sched_setaffinity(0, {core})
            return core
        except (AttributeError, OSError):
            return None

    def __exit__(self, *exc):
        if self.prev:
            os.sched_setaffinity(0, self.prev)
        return False


def run_sweep(args, rank, world):
    """The long-context sweep (Llama-8B GQA shape, 32 q / 8 kv heads): every
    context x batch point at 2 and 4 bits that fits, each its own line."""
    import copy
    import torch
    from bit_kv_cache_kvq_gb300.workloads import SWEEP_BATCHES, SWEEP_CONTEXTS
    for bits in (2, 4):
        for c in SWEEP_CONTEXTS:
            for b in SWEEP_BATCHES:
                a = copy.copy(args)
                a.workload = f"sweep_c{c}_b{b}_k{bits}"
                a.batch = a.context = a.bits = 0
                a.no_e2e = a.no_cpu = True
                a.no_bf16 = args.no_bf16 or bits != 2     # bf16 comparator once per point
                line = run_ours(a, rank, world)
                if rank == 0 and line is not None:
                    print(json.dumps(line), flush=True)
                del line
                torch.cuda.empty_cache()


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    if args.sweep and args.impl == "ours":
        run_sweep(args, rank, world)
    else:
        line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
