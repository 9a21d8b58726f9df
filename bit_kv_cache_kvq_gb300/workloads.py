"""Seeded synthetic inputs with the shapes of the decode workloads.

Recipe: ``torch.randn`` (float32) from a seeded generator, then the outlier
edits of the workload, then one rounding to bf16.  Keys carry a few outlier
channels (a per-KV-head seeded choice applied to all tokens and batch rows:
the QJL page reports about four such key channels in deeper layers; MixKVQ
and KIVI note that values lack them).  The MixKVQ workload's query window
has a few large-|Q| channels.  The pages' own benchmark sets (ShareGPT
through vLLM, LongBench, reasoning suites) are not available; these shapes
stand in for them.

This module holds no quantization, saliency or attention arithmetic.  The
same tensors feed the CUDA path and the CPU oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

D = 128


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    T_q: int              # quantized tokens (prefill length for the prefill workload)
    r: int                # residual tokens
    k_bits: int = 2
    v_bits: int = 2
    k_outliers: int = 4   # outlier key channels per KV head
    k_scale: float = 10.0
    k_shift: float = 0.0
    k_channels: tuple = ()  # fixed outlier channels (tiny workload)
    mode: str = "uniform"
    n_bf16: int = 0
    n_uint4: int = 0
    Lq: int = 0           # query window for saliency
    q_outliers: int = 0
    q_scale: float = 1.0
    steps: int = 0        # decode steps (prefill workload)
    extra: dict = field(default_factory=dict)

    @property
    def n_rep(self) -> int:
        return self.Hq // self.Hkv

    @property
    def T(self) -> int:
        return self.T_q + self.r


WORKLOADS = {
    # single head, 1024 quantized + 64 residual, outlier channels 3 and 77 x8 +20
    "tiny_1head_1k": Workload("tiny_1head_1k", 1001, B=1, Hq=1, Hkv=1, T_q=1024, r=64,
                              k_outliers=0, k_scale=8.0, k_shift=20.0, k_channels=(3, 77)),
    # Llama-3.1-8B decode layer: 32 q / 8 kv heads, batch 16, 32K + 100 residual
    "llama8b_gqa_32k_b16": Workload("llama8b_gqa_32k_b16", 1002, B=16, Hq=32, Hkv=8,
                                    T_q=32768, r=100),
    # prefill 32K at batch 8, then 512 decode steps with a flush every 128
    "llama8b_prefill_32k_b8": Workload("llama8b_prefill_32k_b8", 1003, B=8, Hq=32, Hkv=8,
                                       T_q=32768, r=0, steps=512),
    # KIVI streaming variant (keys in 32-token groups sealed every 128, value
    # FIFO, bf16 metadata) on the Llama-8B decode layer, KIVI-2
    "kivi_llama8b_32k_b16": Workload("kivi_llama8b_32k_b16", 1006, B=16, Hq=32, Hkv=8,
                                     T_q=32768, r=100, mode="kivi"),
    # PN-Mix H3/L1 keys (32 of 64 pairs at 3 bits, the rest 1 bit, adjacent
    # pairs; 2-bit values) on the Llama-8B decode layer; Eq. 6 from a
    # 128-token query window
    "pnmix_llama8b_32k_b16": Workload("pnmix_llama8b_32k_b16", 1007, B=16, Hq=32, Hkv=8,
                                      T_q=32768, r=100, mode="pnmix", Lq=128, q_outliers=8,
                                      q_scale=6.0, extra={"n_high_pairs": 32}),
    # MixKVQ: Qwen-32B layer, 64 q / 8 kv heads, batch 8, 16K context
    "mixkvq_qwen32b_16k_b8": Workload("mixkvq_qwen32b_16k_b8", 1004, B=8, Hq=64, Hkv=8,
                                      T_q=16384, r=100, k_outliers=6, mode="mixed",
                                      n_bf16=6, n_uint4=25, Lq=128, q_outliers=8, q_scale=6.0),
}

SWEEP_CONTEXTS = (4096, 16384, 65536, 131072)
SWEEP_BATCHES = (1, 8, 32, 64)


def sweep_workload(context: int, batch: int, bits: int) -> Workload:
    """Long-context sweep point: Llama-8B GQA shape, T_q = context, r = 100."""
    return Workload(f"sweep_c{context}_b{batch}_k{bits}", 1005, B=batch, Hq=32, Hkv=8,
                    T_q=context, r=100, k_bits=bits, v_bits=bits)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def outlier_channels(seed: int, Hkv: int, n: int) -> torch.Tensor:
    """[Hkv, n] channel ids: the first n of a seeded permutation per KV head."""
    g = _gen(seed, "cpu")
    return torch.stack([torch.randperm(D, generator=g)[:n] for _ in range(Hkv)])


def make_kv(w: Workload, L: int | None = None, device="cpu"):
    """K, V bf16 [B, Hkv, L, D] (L defaults to T_q + r)."""
    L = w.T if L is None else L
    shape = (w.B, w.Hkv, L, D)
    k = torch.randn(shape, generator=_gen(w.seed + 2, device), device=device, dtype=torch.float32)
    if w.k_channels:
        ch = torch.tensor(w.k_channels, device=device)
        k[..., ch] = k[..., ch] * w.k_scale + w.k_shift
    elif w.k_outliers:
        ch = outlier_channels(w.seed + 4, w.Hkv, w.k_outliers).to(device)
        for h in range(w.Hkv):
            k[:, h, :, ch[h]] = k[:, h, :, ch[h]] * w.k_scale + w.k_shift
    k = k.to(torch.bfloat16)
    v = torch.randn(shape, generator=_gen(w.seed + 3, device), device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    return k, v


def make_q(w: Workload, step: int = 0, device="cpu") -> torch.Tensor:
    """Decode query bf16 [B, Hq, D] for a step."""
    return torch.randn((w.B, w.Hq, D), generator=_gen(w.seed + 1 + 1000 * step, device),
                       device=device, dtype=torch.float32).to(torch.bfloat16)


def make_token(w: Workload, step: int, device="cpu"):
    """New key/value of one decode step, bf16 [B, Hkv, D] each (same outlier
    channels as the history)."""
    k = torch.randn((w.B, w.Hkv, D), generator=_gen(w.seed + 5 + 1000 * step, device),
                    device=device, dtype=torch.float32)
    if w.k_channels:
        ch = torch.tensor(w.k_channels, device=device)
        k[..., ch] = k[..., ch] * w.k_scale + w.k_shift
    elif w.k_outliers:
        ch = outlier_channels(w.seed + 4, w.Hkv, w.k_outliers).to(device)
        for h in range(w.Hkv):
            k[:, h, ch[h]] = k[:, h, ch[h]] * w.k_scale + w.k_shift
    v = torch.randn((w.B, w.Hkv, D), generator=_gen(w.seed + 6 + 1000 * step, device),
                    device=device, dtype=torch.float32)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def make_query_window(w: Workload, device="cpu") -> torch.Tensor:
    """MixKVQ query window bf16 [B, Hq, Lq, D] with q_outliers channels x q_scale."""
    q = torch.randn((w.B, w.Hq, w.Lq, D), generator=_gen(w.seed + 7, device), device=device,
                    dtype=torch.float32)
    if w.q_outliers:
        ch = outlier_channels(w.seed + 8, 1, w.q_outliers)[0].to(device)
        q[..., ch] = q[..., ch] * w.q_scale
    return q.to(torch.bfloat16)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(changes)
    return Workload(**d)


def bf16_bits(t: torch.Tensor):
    """Raw bf16 patterns of a bf16 tensor as a numpy uint16 array (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
