"""CPU checks of the C ABI: libkvq.so builds, loads without a GPU, exports
every function include/kvq.h declares, and its host-side byte accounting
matches the oracle's (pinned to the KIVI article's §7 formula)."""
import ctypes
import os
import re

import pytest

import oracle as orc
from bit_kv_cache_kvq_gb300 import _build
import bit_kv_cache_kvq_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kvq.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kvq_cache_alloc", "kvq_append_residual", "kvq_flush_group",
                     "kvq_quantize_prefill", "kvq_decode_attention", "kvq_channel_saliency"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libkvq.so does not export {name}"


def _bytes(B, Hkv, T, k_bits=2, v_bits=2, mode=0, nb=0, n4=0, D=128):
    cfg = kvq._Config(B, Hkv, D, T, k_bits, v_bits, mode, nb, n4)
    return kvq.lib().kvq_cache_bytes(ctypes.byref(cfg))


@pytest.mark.parametrize("k_bits,v_bits", [(2, 2), (4, 4), (2, 4), (4, 2)])
def test_record_bytes_match_oracle_accounting(lib, k_bits, v_bits):
    """Per 128-token group of one (b, kv head): codes at b/8 bytes per
    element, a bf16 origin and an fp32 step per Key channel group (128
    tokens) and per Value token group (32 channels)."""
    per_group = (_bytes(1, 1, 128 * 9, k_bits, v_bits) - _bytes(1, 1, 128, k_bits, v_bits)) / 8
    ref = orc.cache_bytes(T=128, rK=0, rV=0, D=128, k_bits=k_bits, v_bits=v_bits, Gk=128,
                          Gv=32, origin_bytes=2, step_bytes=4, float_bytes=2)
    assert per_group == ref
    assert ref / 128 == {(2, 2): 94, (4, 4): 158, (2, 4): 126, (4, 2): 126}[(k_bits, v_bits)]


def test_mixed_record_bytes(lib):
    """Mixed keys, 6 BF16 / 25 UINT4 / 97 UINT2 channels: channel permutation
    (128 B) + raw bf16 + 4-bit and 2-bit codes + (fp32 step, bf16 origin) per
    quantized channel = 7100 B.  Stored as 2-bit virtual channels (two per
    UINT4 channel): 147, zero-padded to 160 (13 x 32 B), then to a 128-byte
    line; values as uniform 2-bit."""
    per_group = (_bytes(1, 1, 128 * 9, 2, 2, 1, 6, 25) - _bytes(1, 1, 128, 2, 2, 1, 6, 25)) / 8
    kpart = 128 + 6 * 128 * 2 + 25 * 64 + 97 * 32 + (25 + 97) * 6
    assert kpart == 7100
    padding = (160 - (2 * 25 + 97)) * 32
    v = orc.cache_bytes(T=128, rK=128, rV=0, D=128, k_bits=2, v_bits=2, Gk=128, Gv=32,
                        origin_bytes=2, step_bytes=4, float_bytes=0)
    assert per_group == (kpart + padding + 127) // 128 * 128 + v


def test_sink_windows_add_their_bytes(lib):
    """An attention-sink window of n_sink tokens adds two bf16 windows
    [B][Hkv][n_sink][D] (rounded to 256 bytes)."""
    base = _bytes(2, 3, 256)
    cfg = kvq._Config(2, 3, 128, 256, 2, 2, 0, 0, 0, 32)
    with_sink = kvq.lib().kvq_cache_bytes(ctypes.byref(cfg))
    assert with_sink - base == 2 * ((2 * 3 * 32 * 128 * 2 + 255) // 256 * 256)


def test_invalid_configs_report_zero_bytes(lib):
    assert _bytes(1, 1, 128, D=64) == 0          # head_dim other than 128
    assert _bytes(1, 1, 100) == 0                # capacity not a multiple of 128
    assert _bytes(1, 1, 128, k_bits=3) == 0
    assert _bytes(0, 1, 128) == 0
    assert _bytes(1, 1, 128, mode=1, nb=100, n4=40) == 0
    for n_sink in (-1, 129):                     # sink window 0..128
        cfg = kvq._Config(1, 1, 128, 128, 2, 2, 0, 0, 0, n_sink)
        assert kvq.lib().kvq_cache_bytes(ctypes.byref(cfg)) == 0


def test_status_strings(lib):
    lib.kvq_status_string.restype = ctypes.c_char_p
    assert lib.kvq_status_string(0) == b"KVQ_OK"
    assert lib.kvq_status_string(4) == b"KVQ_ERR_RESIDUAL_FULL"
