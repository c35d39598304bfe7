"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/kvq.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def K():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "kvq_build", os.path.join(ROOT, "quantized_paged_kv_quantize_gb300", "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    from quantized_paged_kv_quantize_gb300 import kvq
    return kvq


def test_exports_every_declared_function(K):
    names = _header_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(K.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in kvq.h but not exported"
    assert set(names) == set(K.EXPORTED)


def test_version_and_sizes(K):
    assert K.kvq_version() == 1
    # bytes per (page, kv head) block: the documented layout
    assert K.kvq_cache_block_bytes(K.make_config(1, 16, 1, 128, "fp8_per_tensor")) == 4096
    assert K.kvq_cache_block_bytes(K.make_config(1, 16, 1, 128, "int8_per_token_head")) == 4224
    assert K.kvq_cache_block_bytes(K.make_config(1, 16, 1, 128, "fp8_per_token_head")) == 4224
    assert K.kvq_cache_block_bytes(K.make_config(1, 16, 1, 128, "nvfp4")) == 2304
    assert K.kvq_cache_block_bytes(K.make_config(1, 16, 1, 128, "nvfp4_4over6")) == 2304
    assert K.kvq_cache_block_bytes(K.make_config(1, 16, 1, 128, "int4_per_token_head")) == 2176
    assert K.kvq_cache_block_bytes(K.make_config(1, 128, 1, 128, "kvarn_k4v2_g128")) == 16384
    assert K.kvq_cache_bytes(K.make_config(10, 16, 8, 128, "nvfp4")) == 256 + 10 * 8 * 2304


def test_layout_matches_oracle(K):
    import oracle
    for mode in ("fp8_per_tensor", "int8_per_token_head", "fp8_per_token_head", "nvfp4", "int4_per_token_head",
                 "nvfp4_4over6"):
        for D in (32, 128):
            cfg = K.make_config(7, 16, 3, D, mode)
            assert K.kvq_cache_bytes(cfg) == oracle.pool_bytes(mode, 7, 16, 3, D)
    assert K.kvq_cache_bytes(K.make_config(5, 128, 2, 128, "kvarn_k4v2_g128")) == \
        oracle.pool_bytes("kvarn_k4v2_g128", 5, 128, 2, 128)


@pytest.mark.parametrize("args,status", [
    ((4, 16, 2, 64, "nvfp4"), 2),             # head_dim 64
    ((4, 32, 2, 128, "nvfp4"), 2),            # page 32
    ((4, 16, 2, 128, "kvarn_k4v2_g128"), 2),  # kvarn needs page 128
    ((4, 128, 2, 64, "kvarn_k4v2_g128"), 2),  # kvarn needs D 128
    ((0, 16, 2, 128, "nvfp4"), 1),            # no pages
    ((4, 16, 0, 128, "nvfp4"), 1),            # no heads
    ((4, 16, 2, 128, 9), 2),                  # unknown mode
])
def test_config_rejected(K, args, status):
    with pytest.raises(K.KVQError) as e:
        K.kvq_cache_bytes(K.make_config(*args))
    assert e.value.status == status


def test_bad_pointers_rejected_before_device_work(K):
    lib = K.lib()
    cfg = K.make_config(4, 16, 2, 128, "nvfp4")
    h = ctypes.c_void_p()
    assert lib.kvq_cache_alloc(ctypes.byref(cfg), None, 1 << 20, ctypes.byref(h)) == 1
    assert lib.kvq_cache_alloc(ctypes.byref(cfg), 0x1001, 1 << 20, ctypes.byref(h)) == 1   # misaligned
    assert lib.kvq_cache_alloc(ctypes.byref(cfg), 0x100000, 16, ctypes.byref(h)) == 4      # too small
    assert b"bytes" in lib.kvq_last_error()
    assert lib.kvq_quantize_write(None, None, None, None, 1, 4, None) == 1
    assert lib.kvq_decode_attention(None, None, None, 0, None, 1, 8, 16, 4, 0.1, None, 0, None, 0, None) == 1
    assert lib.kvq_tensor_amax(None, 0, 5, None, None) == 1
    assert lib.kvq_tensor_amax(None, 7, 5, None, None) == 2
    assert lib.kvq_cache_free(None) == 0
