"""CPU checks of the C ABI: the library loads and exports every declared entry."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvint2.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:kv_status_t|size_t)\s+(kv_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def built_lib():
    from bit_kv_cache_12_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_hot_path_entries():
    names = declared_functions()
    for required in ["kv_pool_create", "kv_append_quantize", "kv_append_step", "kv_decode_attention",
                     "kv_decode_attention_bf16", "kv_quantize_pack_f32"]:
        assert required in names


def test_library_exports_every_declared_symbol(built_lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(built_lib, n), n


def test_binding_signatures_cover_the_header():
    from bit_kv_cache_12_gb300 import native
    assert set(declared_functions()) == set(native._SIG)


def test_invalid_arguments_rejected_without_gpu(built_lib):
    """Host-side validation runs before any CUDA call."""
    from bit_kv_cache_12_gb300 import native
    L = native.lib()
    assert L.kv_pool_create(None, None, None) == native.KV_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    cfg = native.KvPoolConfig(0, 1, 8, 2, 64, 16, 128, 64, 256, 1, 10)      # head_dim 64
    assert L.kv_pool_create(ctypes.byref(cfg), None, ctypes.byref(h)) == native.KV_ERR_UNSUPPORTED
    cfg = native.KvPoolConfig(0, 1, 8, 3, 128, 16, 128, 64, 256, 1, 10)     # Hq % Hkv != 0
    assert L.kv_pool_create(ctypes.byref(cfg), None, ctypes.byref(h)) == native.KV_ERR_INVALID_ARG
    cfg = native.KvPoolConfig(0, 1, 8, 2, 128, 8, 128, 64, 256, 1, 10)      # page 8
    assert L.kv_pool_create(ctypes.byref(cfg), None, ctypes.byref(h)) == native.KV_ERR_UNSUPPORTED
    cfg = native.KvPoolConfig(0, 1, 8, 2, 128, 16, 32, 64, 256, 1, 10)      # group 32
    assert L.kv_pool_create(ctypes.byref(cfg), None, ctypes.byref(h)) == native.KV_ERR_UNSUPPORTED
    assert L.kv_decode_attention(None, 0, 1, None, None, None, None, None, None, 1, 0,
                                 ctypes.c_float(1.0), None, None, 0, None) == native.KV_ERR_INVALID_ARG
    assert L.kv_decode_workspace_bytes(None, 1, 100) == 0
    assert L.kv_append_step(None, 0, 1, None, None, None, None, None, None, None, 1,
                            None) == native.KV_ERR_INVALID_ARG


def test_binding_has_a_wrapper_for_every_entry():
    from bit_kv_cache_12_gb300 import native
    for name in native._SIG:
        assert callable(getattr(native, name, None)), name
