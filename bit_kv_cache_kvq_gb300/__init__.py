"""GB300 low-bit KV-cache quantization and fused decode attention.

Thin ctypes binding over ``libkvq.so`` (declared in ``include/kvq.h``).  Every
computation runs in the library's CUDA kernels; this module only checks
tensor dtypes/shapes/devices, passes raw pointers and the current CUDA stream,
and turns return codes into exceptions.  PyTorch provides device memory and
streams.  There is no CPU fallback: if the library is missing the first call
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "KVCache", "decode_bf16", "channel_saliency", "KVQError", "lib",
    "KVQ_K_UNIFORM", "KVQ_K_MIXED", "KVQ_K_KIVI", "KVQ_K_PNMIX", "TIER_BF16", "TIER_UINT4", "TIER_UINT2",
    "FLAG_NONFINITE", "FLAG_RANGE", "FLAG_TIMEOUT", "set_wait_limit", "HEAD_DIM", "K_GROUP", "V_GROUP", "RESIDUAL",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

HEAD_DIM, K_GROUP, V_GROUP, RESIDUAL = 128, 128, 32, 128
KVQ_K_UNIFORM, KVQ_K_MIXED, KVQ_K_KIVI, KVQ_K_PNMIX = 0, 1, 2, 3
_MODES = {"uniform": KVQ_K_UNIFORM, "mixed": KVQ_K_MIXED, "kivi": KVQ_K_KIVI,
          "pnmix": KVQ_K_PNMIX}
PAIRS_ADJACENT, PAIRS_SPLIT = 0, 1
TIER_BF16, TIER_UINT4, TIER_UINT2 = 0, 1, 2
TIERS_RANK, TIERS_THRESHOLD = 0, 1
FLAG_NONFINITE, FLAG_RANGE, FLAG_TIMEOUT = 1, 2, 4

_CODES = {0: "OK", 1: "ARG", 2: "SHAPE", 3: "CAPACITY", 4: "RESIDUAL_FULL",
          5: "RESIDUAL_NOT_FULL", 6: "EMPTY", 7: "NOT_EMPTY", 8: "CUDA", 9: "WORKSPACE",
          10: "MODE"}


class KVQError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: KVQ_ERR_{_CODES.get(code, code)}")
        self.code = code
        self.name = _CODES.get(code, str(code))


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "kv_heads", "head_dim", "max_tokens", "k_bits", "v_bits", "k_mode",
        "n_bf16", "n_uint4", "n_sink", "tier_mode")] + [
        ("tau_bf16", ctypes.c_float), ("tau_uint4", ctypes.c_float),
        ("n_high_pairs", ctypes.c_int), ("pair_layout", ctypes.c_int)]


class _TierSpec(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("n_bf16", ctypes.c_int), ("n_uint4", ctypes.c_int),
                ("tau_bf16", ctypes.c_float), ("tau_uint4", ctypes.c_float)]


_lib = None

# name -> (restype, argtypes); P = pointer, I = int, Z = size_t
_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "kvq_cache_bytes": (_Z, [_P]),
    "kvq_cache_alloc": (_I, [_P, _P, _Z, _P, _P]),
    "kvq_cache_free": (_I, [_P, _P]),
    "kvq_cache_lengths": (_I, [_P, _P, _P]),
    "kvq_cache_sink_tokens": (_I, [_P, _P]),
    "kvq_cache_reset": (_I, [_P, _P]),
    "kvq_append_residual": (_I, [_P, _P, _P, _P]),
    "kvq_flush_group": (_I, [_P, _P, _P]),
    "kvq_observe_query": (_I, [_P, _P, _I, _P]),
    "kvq_quantize_prefill": (_I, [_P, _P, _P, _I, _P, _P]),
    "kvq_decode_workspace_bytes": (_Z, [_P, _I]),
    "kvq_decode_step": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _Z, _P]),
    "kvq_decode_attention": (_I, [_P, _P, _I, _P, _P, _Z, _P]),
    "kvq_decode_bf16_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "kvq_decode_bf16": (_I, [_P, _P, _I, _I, _I, _P, _I, _P, _P, _Z, _P]),
    "kvq_channel_saliency": (_I, [_P, _I, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "kvq_cache_status": (_I, [_P, _P, _P]),
    "kvq_export_k": (_I, [_P, _P, _P, _P, _P]),
    "kvq_export_v": (_I, [_P, _P, _P, _P, _P]),
    "kvq_export_residual": (_I, [_P, _P, _P, _P]),
    "kvq_export_sink": (_I, [_P, _P, _P, _P]),
    "kvq_export_k_mixed": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "kvq_set_wait_limit": (_I, [_I]),
    "kvq_set_decode_split_event": (_I, [_P]),
    "kvq_export_kivi": (_I, [_P] * 10),
    "kvq_pnmix_pairs": (_I, [_P, _P, _I, _I, _P, _I, _P, _P]),
    "kvq_export_pnmix": (_I, [_P] * 6),
    "kvq_status_string": (ctypes.c_char_p, [_I]),
}


def lib() -> ctypes.CDLL:
    """Load libkvq.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvq.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(code: int, what: str):
    if code != 0:
        raise KVQError(code, what)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None, dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    # one combined test on the common path (a decode step checks seven tensors)
    if (t.is_cuda and (dtype is None or t.dtype == dtype)
            and (shape is None or t.shape == shape) and t.is_contiguous()):
        return t.data_ptr()
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class KVCache:
    """One layer's packed KV cache on the current GPU (MixKVQ Algorithm 1
    state: packed history + bf16 residual of up to 128 tokens).

    mode "uniform": keys at k_bits per channel over 128-token groups;
    mode "mixed": keys tiered per group into BF16, UINT4 and UINT2 channels,
    tier_mode "rank" exactly n_bf16 / n_uint4 of the first two, "threshold"
    A > tau_bf16 / A > tau_uint4 with at most n_bf16 / n_uint4 of them.
    Values always v_bits per token over 32 channels.
    n_sink > 0 keeps the sequence's first n_sink tokens bf16 (attention
    sinks, never quantized).
    The device buffer is a torch uint8 tensor owned by this object.
    """

    def __init__(self, batch: int, kv_heads: int, max_tokens: int, k_bits: int = 2,
                 v_bits: int = 2, mode: str = "uniform", n_bf16: int = 0, n_uint4: int = 0,
                 head_dim: int = HEAD_DIM, device=None, stream=None, n_sink: int = 0,
                 tier_mode: str = "rank", tau_bf16: float = 0.0, tau_uint4: float = 0.0,
                 n_high_pairs: int = 0, pair_layout: int = PAIRS_ADJACENT):
        if tier_mode not in ("rank", "threshold"):
            raise ValueError("tier_mode is 'rank' or 'threshold'")
        if mode not in _MODES:
            raise ValueError("mode is 'uniform', 'mixed', 'kivi' or 'pnmix'")
        self.cfg = _Config(batch, kv_heads, head_dim, max_tokens, k_bits, v_bits,
                           _MODES[mode], n_bf16, n_uint4,
                           n_sink, TIERS_THRESHOLD if tier_mode == "threshold"
                           else TIERS_RANK, tau_bf16, tau_uint4, n_high_pairs, pair_layout)
        self.tier_mode = tier_mode
        self.mode = mode
        nbytes = lib().kvq_cache_bytes(ctypes.byref(self.cfg))
        if nbytes == 0:
            raise KVQError(1, "kvq_cache_bytes (invalid config)")
        self.nbytes = nbytes
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            _check(lib().kvq_cache_alloc(ctypes.byref(self.cfg), self.buffer.data_ptr(), nbytes,
                                         _stream(stream), ctypes.byref(h)), "kvq_cache_alloc")
        self._h = h
        self.batch, self.kv_heads, self.max_tokens = batch, kv_heads, max_tokens
        self.k_bits, self.v_bits, self.n_bf16, self.n_uint4 = k_bits, v_bits, n_bf16, n_uint4
        self.n_sink = n_sink
        self.device = dev

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.kvq_cache_free(h, None)
            self._h = None

    @property
    def handle(self):
        return self._h

    # -- state
    def lengths(self) -> tuple[int, int]:
        tq, r = ctypes.c_int(), ctypes.c_int()
        _check(lib().kvq_cache_lengths(self._h, ctypes.byref(tq), ctypes.byref(r)), "lengths")
        return tq.value, r.value

    def sink_tokens(self) -> int:
        s = ctypes.c_int()
        _check(lib().kvq_cache_sink_tokens(self._h, ctypes.byref(s)), "sink_tokens")
        return s.value

    def status(self, stream=None) -> int:
        st = ctypes.c_int()
        _check(lib().kvq_cache_status(self._h, _stream(stream), ctypes.byref(st)), "status")
        return st.value

    def reset(self, stream=None):
        _check(lib().kvq_cache_reset(self._h, _stream(stream)), "reset")

    # -- Algorithm 1
    def prefill(self, k: torch.Tensor, v: torch.Tensor, importance: torch.Tensor | None = None,
                stream=None):
        B, H, L, D = k.shape
        shp = (self.batch, self.kv_heads, L, HEAD_DIM)
        _check(lib().kvq_quantize_prefill(
            self._h, _ptr(k, torch.bfloat16, shp, "k"), _ptr(v, torch.bfloat16, shp, "v"), L,
            _ptr(importance, torch.float32, (self.batch, self.kv_heads, HEAD_DIM), "importance"),
            _stream(stream)), "kvq_quantize_prefill")

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        shp = (self.batch, self.kv_heads, HEAD_DIM)
        _check(lib().kvq_append_residual(self._h, _ptr(k_new, torch.bfloat16, shp, "k_new"),
                                         _ptr(v_new, torch.bfloat16, shp, "v_new"),
                                         _stream(stream)), "kvq_append_residual")

    def observe(self, q: torch.Tensor, stream=None):
        """Add one decode step's query (bf16 [B, Hq, D]) to the mixed cache's
        online |q| window (the importance a flush without one uses)."""
        B, Hq, D = q.shape
        _check(lib().kvq_observe_query(self._h, _ptr(q, torch.bfloat16, (self.batch, Hq, HEAD_DIM),
                                                     "q"), Hq, _stream(stream)),
               "kvq_observe_query")

    def flush(self, importance: torch.Tensor | None = None, stream=None):
        _check(lib().kvq_flush_group(
            self._h, _ptr(importance, torch.float32, (self.batch, self.kv_heads, HEAD_DIM),
                          "importance"), _stream(stream)), "kvq_flush_group")

    def workspace_bytes(self, Hq: int) -> int:
        return lib().kvq_decode_workspace_bytes(self._h, Hq)

    def workspace(self, Hq: int) -> torch.Tensor:
        return torch.empty(self.workspace_bytes(Hq), dtype=torch.uint8, device=self.device)

    def attention(self, q: torch.Tensor, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        B, Hq, D = q.shape
        if out is None:
            out = torch.empty(B, Hq, HEAD_DIM, dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = self.workspace(Hq)
        _check(lib().kvq_decode_attention(
            self._h, _ptr(q, torch.bfloat16, (self.batch, Hq, HEAD_DIM), "q"), Hq,
            _ptr(out, torch.float32, (self.batch, Hq, HEAD_DIM), "out"),
            _ptr(workspace, torch.uint8, None, "workspace"), workspace.numel(),
            _stream(stream)), "kvq_decode_attention")
        return out

    def decode_step(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    importance: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Append the token, flush if the residual is full, attend (one call,
        kvq_decode_step)."""
        B, Hq, D = q.shape
        if out is None:
            out = torch.empty(B, Hq, HEAD_DIM, dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = self.workspace(Hq)
        shp = (self.batch, self.kv_heads, HEAD_DIM)
        _check(lib().kvq_decode_step(
            self._h, _ptr(k_new, torch.bfloat16, shp, "k_new"),
            _ptr(v_new, torch.bfloat16, shp, "v_new"),
            _ptr(importance, torch.float32, shp, "importance"),
            _ptr(q, torch.bfloat16, (self.batch, Hq, HEAD_DIM), "q"), Hq,
            _ptr(out, torch.float32, (self.batch, Hq, HEAD_DIM), "out"),
            _ptr(workspace, torch.uint8, None, "workspace"), workspace.numel(),
            _stream(stream)), "kvq_decode_step")
        return out

    # -- canonical export (device tensors)
    def export_k(self, stream=None):
        tq, _ = self.lengths()
        n = tq // K_GROUP
        B, H, dev = self.batch, self.kv_heads, self.device
        codes = torch.empty(B, H, n, HEAD_DIM, K_GROUP * self.k_bits // 8, dtype=torch.uint8, device=dev)
        kmin = torch.empty(B, H, n, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        kscale = torch.empty(B, H, n, HEAD_DIM, dtype=torch.float32, device=dev)
        _check(lib().kvq_export_k(self._h, codes.data_ptr(), kmin.data_ptr(), kscale.data_ptr(),
                                  _stream(stream)), "kvq_export_k")
        return codes, kmin, kscale

    def export_v(self, stream=None):
        tq, _ = self.lengths()
        B, H, dev = self.batch, self.kv_heads, self.device
        codes = torch.empty(B, H, tq, HEAD_DIM * self.v_bits // 8, dtype=torch.uint8, device=dev)
        vmin = torch.empty(B, H, tq, HEAD_DIM // V_GROUP, dtype=torch.bfloat16, device=dev)
        vscale = torch.empty(B, H, tq, HEAD_DIM // V_GROUP, dtype=torch.float32, device=dev)
        _check(lib().kvq_export_v(self._h, codes.data_ptr(), vmin.data_ptr(), vscale.data_ptr(),
                                  _stream(stream)), "kvq_export_v")
        return codes, vmin, vscale

    def export_residual(self, stream=None):
        _, r = self.lengths()
        B, H, dev = self.batch, self.kv_heads, self.device
        kr = torch.empty(B, H, r, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        vr = torch.empty(B, H, r, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        _check(lib().kvq_export_residual(self._h, kr.data_ptr(), vr.data_ptr(), _stream(stream)),
               "kvq_export_residual")
        return kr, vr

    def export_sink(self, stream=None):
        s = self.sink_tokens()
        B, H, dev = self.batch, self.kv_heads, self.device
        ks = torch.empty(B, H, s, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        vs = torch.empty(B, H, s, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        _check(lib().kvq_export_sink(self._h, ks.data_ptr(), vs.data_ptr(), _stream(stream)),
               "kvq_export_sink")
        return ks, vs

    def pnmix_pairs(self, q: torch.Tensor, k: torch.Tensor, stream=None) -> torch.Tensor:
        """PN-Mix Eq. 6 pair scores from the prefill queries q bf16 [B, Hq, Lq,
        D] and keys k bf16 [B, Hkv, Lk, D]; the cache keeps the selection of
        n_high_pairs pairs.  Returns sigma fp32 [B, Hkv, D/2]."""
        B, Hq, Lq, D = q.shape
        Lk = k.shape[2]
        sigma = torch.empty(self.batch, self.kv_heads, HEAD_DIM // 2, dtype=torch.float32,
                            device=q.device)
        _check(lib().kvq_pnmix_pairs(
            self._h, _ptr(q, torch.bfloat16, (self.batch, Hq, Lq, HEAD_DIM), "q"), Hq, Lq,
            _ptr(k, torch.bfloat16, (self.batch, self.kv_heads, Lk, HEAD_DIM), "k"), Lk,
            sigma.data_ptr(), _stream(stream)), "kvq_pnmix_pairs")
        return sigma

    def export_pnmix(self, stream=None):
        """PN-Mix key groups (kvq_export_pnmix): codes uint8 [B, Hkv, n, 128, D],
        offset / scale fp32 [B, Hkv, n, D], high uint8 [B, Hkv, D]."""
        tq, _ = self.lengths()
        n = tq // K_GROUP
        B, H, dev = self.batch, self.kv_heads, self.device
        codes = torch.zeros(B, H, n, K_GROUP, HEAD_DIM, dtype=torch.uint8, device=dev)
        off = torch.zeros(B, H, n, HEAD_DIM, dtype=torch.float32, device=dev)
        sc = torch.zeros(B, H, n, HEAD_DIM, dtype=torch.float32, device=dev)
        high = torch.zeros(B, H, HEAD_DIM, dtype=torch.uint8, device=dev)
        ptr = lambda t: t.data_ptr() if t.numel() else None
        _check(lib().kvq_export_pnmix(self._h, ptr(codes), ptr(off), ptr(sc), high.data_ptr(),
                                      _stream(stream)), "kvq_export_pnmix")
        return codes, off, sc, high

    def export_kivi(self, stream=None):
        """KIVI cache state (kvq_export_kivi): dict of device tensors k_codes
        [B, Hkv, n*4, D, 32*bits/8], k_origin/k_step bf16 [B, Hkv, n*4, D],
        v_codes [B, Hkv, n*128, D*bits/8], v_origin/v_step bf16 [B, Hkv,
        n*128, D/32], k_res [B, Hkv, r_K, D], v_res [B, Hkv, r_V, D] (FIFO,
        oldest first); n = T_k / 128."""
        tk, rk = self.lengths()
        n, rv = tk // K_GROUP, min(tk + rk, RESIDUAL)
        B, H, dev, b = self.batch, self.kv_heads, self.device, self.k_bits
        out = {
            "k_codes": torch.zeros(B, H, n * 4, HEAD_DIM, 32 * b // 8, dtype=torch.uint8, device=dev),
            "k_origin": torch.zeros(B, H, n * 4, HEAD_DIM, dtype=torch.bfloat16, device=dev),
            "k_step": torch.zeros(B, H, n * 4, HEAD_DIM, dtype=torch.bfloat16, device=dev),
            "v_codes": torch.zeros(B, H, n * 128, HEAD_DIM * self.v_bits // 8, dtype=torch.uint8,
                                   device=dev),
            "v_origin": torch.zeros(B, H, n * 128, HEAD_DIM // V_GROUP, dtype=torch.bfloat16, device=dev),
            "v_step": torch.zeros(B, H, n * 128, HEAD_DIM // V_GROUP, dtype=torch.bfloat16, device=dev),
            "k_res": torch.zeros(B, H, rk, HEAD_DIM, dtype=torch.bfloat16, device=dev),
            "v_res": torch.zeros(B, H, rv, HEAD_DIM, dtype=torch.bfloat16, device=dev),
        }
        ptr = lambda t: t.data_ptr() if t.numel() else None
        _check(lib().kvq_export_kivi(self._h, *(ptr(out[k]) for k in (
            "k_codes", "k_origin", "k_step", "v_codes", "v_origin", "v_step", "k_res", "v_res")),
            _stream(stream)), "kvq_export_kivi")
        return out

    def export_k_mixed(self, stream=None):
        tq, _ = self.lengths()
        n = tq // K_GROUP
        B, H, dev = self.batch, self.kv_heads, self.device
        nb, n4 = self.n_bf16, self.n_uint4
        n2 = HEAD_DIM if self.tier_mode == "threshold" else HEAD_DIM - nb - n4
        t = dict(
            counts=torch.empty(B, H, n, 2, dtype=torch.uint8, device=dev),
            perm=torch.empty(B, H, n, HEAD_DIM, dtype=torch.uint8, device=dev),
            raw=torch.empty(B, H, n, nb, K_GROUP, dtype=torch.bfloat16, device=dev),
            c4=torch.empty(B, H, n, n4, K_GROUP // 2, dtype=torch.uint8, device=dev),
            m4=torch.empty(B, H, n, n4, dtype=torch.bfloat16, device=dev),
            s4=torch.empty(B, H, n, n4, dtype=torch.float32, device=dev),
            c2=torch.empty(B, H, n, n2, K_GROUP // 4, dtype=torch.uint8, device=dev),
            m2=torch.empty(B, H, n, n2, dtype=torch.bfloat16, device=dev),
            s2=torch.empty(B, H, n, n2, dtype=torch.float32, device=dev))
        _check(lib().kvq_export_k_mixed(self._h, *[x.data_ptr() for x in t.values()],
                                        _stream(stream)), "kvq_export_k_mixed")
        return t


def decode_bf16(k: torch.Tensor, v: torch.Tensor, q: torch.Tensor,
                out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Unquantized comparator over bf16 k, v [B, Hkv, T, D]; q [B, Hq, D]."""
    B, Hkv, T, D = k.shape
    Hq = q.shape[1]
    if out is None:
        out = torch.empty(B, Hq, HEAD_DIM, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(lib().kvq_decode_bf16_workspace_bytes(B, Hkv, T, Hq),
                                dtype=torch.uint8, device=q.device)
    _check(lib().kvq_decode_bf16(
        _ptr(k, torch.bfloat16, (B, Hkv, T, HEAD_DIM), "k"),
        _ptr(v, torch.bfloat16, (B, Hkv, T, HEAD_DIM), "v"), B, Hkv, T,
        _ptr(q, torch.bfloat16, (B, Hq, HEAD_DIM), "q"), Hq,
        _ptr(out, torch.float32, (B, Hq, HEAD_DIM), "out"),
        _ptr(workspace, torch.uint8, None, "workspace"), workspace.numel(), _stream(stream)),
        "kvq_decode_bf16")
    return out


def channel_saliency(q_win: torch.Tensor, k_grp: torch.Tensor, sal_bits: int = 2,
                     n_bf16: int | None = None, n_uint4: int | None = None,
                     tau_bf16: float | None = None, tau_uint4: float | None = None,
                     stream=None):
    """MixKVQ I_d, A_d = I_d * S_d and tiers per (b, kv head, d).

    q_win bf16 [B, Hq, Lq, D]; k_grp bf16 [B, Hkv, G, D].  Rank tiers when
    n_bf16/n_uint4 are given, threshold tiers when tau_bf16/tau_uint4 are.
    Returns (I, A, tiers) as device tensors.
    """
    B, Hq, Lq, D = q_win.shape
    _, Hkv, G, _ = k_grp.shape
    if n_bf16 is not None:
        spec = _TierSpec(TIERS_RANK, n_bf16, n_uint4 or 0, 0.0, 0.0)
    else:
        spec = _TierSpec(TIERS_THRESHOLD, 0, 0, float(tau_bf16), float(tau_uint4))
    dev = q_win.device
    I = torch.empty(B, Hkv, HEAD_DIM, dtype=torch.float32, device=dev)
    A = torch.empty_like(I)
    tiers = torch.empty(B, Hkv, HEAD_DIM, dtype=torch.uint8, device=dev)
    _check(lib().kvq_channel_saliency(
        _ptr(q_win, torch.bfloat16, (B, Hq, Lq, HEAD_DIM), "q_win"), Hq, Lq,
        _ptr(k_grp, torch.bfloat16, (B, Hkv, G, HEAD_DIM), "k_grp"), B, Hkv, G, sal_bits,
        ctypes.byref(spec), I.data_ptr(), A.data_ptr(), tiers.data_ptr(), _stream(stream)),
        "kvq_channel_saliency")
    return I, A, tiers


def set_wait_limit(polls: int) -> int:
    """Polls before a decode warp's wait for its staged data gives up
    (kvq_set_wait_limit; negative restores the default).  A failure-detection
    hook for tests: 0 makes every wait give up at once, setting
    FLAG_TIMEOUT.  Returns the previous limit."""
    return int(lib().kvq_set_wait_limit(int(polls)))


def set_decode_split_event(event) -> None:
    """The next decode attention call records ``event`` (a
    ``torch.cuda.Event`` with timing, or None to cancel) between its decode
    kernel and its combine (kvq_set_decode_split_event): an event recorded
    before the call and this one bracket the decode kernel alone."""
    if event is not None and not event.cuda_event:
        event.record()   # torch creates its events on their first record
    handle = None if event is None else ctypes.c_void_p(int(event.cuda_event))
    _check(lib().kvq_set_decode_split_event(handle), "kvq_set_decode_split_event")
