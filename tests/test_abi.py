"""The C-ABI library loads without a GPU and exports every entry point that
include/moecache.h declares (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moecache.h")
LIB = os.path.join(ROOT, "expert_cache_serving_gb300", "_lib", "libmoecache.so")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_cache_create", "moe_cache_resize", "moe_layer_forward", "moe_prefill_stream",
                     "moe_cache_destroy", "moe_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol():
    if not os.path.exists(LIB):
        pytest.skip("library not built")
    lib = ctypes.CDLL(LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_matches_header():
    if not os.path.exists(LIB):
        pytest.skip("library not built")
    from expert_cache_serving_gb300 import moecache as mc

    assert sorted(mc.SIGNATURES) == declared_functions()
    assert mc.moe_version() == 1


def test_host_side_validation_without_gpu():
    if not os.path.exists(LIB):
        pytest.skip("library not built")
    from expert_cache_serving_gb300 import moecache as mc

    good = mc.moe_model_desc(2, 16, 2, 256, 128, mc.MOE_FP32, 0, 1)
    assert mc.moe_record_bytes(good) == 12 * 256 * 128
    assert mc.moe_record_bytes(mc.moe_model_desc(40, 256, 8, 2048, 512, mc.MOE_BF16, 1, 1)) == 6291456
    assert mc.moe_record_bytes(mc.moe_model_desc(43, 256, 6, 4096, 2048, mc.MOE_FP4, 0, 8)) == 14155776
    for bad in [mc.moe_model_desc(2, 16, 17, 256, 128, 0, 0, 1),    # k > E
                mc.moe_model_desc(2, 2048, 2, 256, 128, 0, 0, 1),   # E too large
                mc.moe_model_desc(2, 16, 2, 100, 128, 0, 0, 1),     # H not a multiple of 64
                mc.moe_model_desc(2, 16, 2, 256, 128, 2, 0, 1),     # FP4 needs multiples of 256
                mc.moe_model_desc(2, 16, 2, 256, 128, 0, 0, 17),    # max_tokens > 16
                mc.moe_model_desc(2, 16, 2, 256, 128, 5, 0, 1)]:    # unknown format
        assert mc.moe_record_bytes(bad) == 0
    out = ctypes.c_void_p()
    st = mc.lib.moe_cache_create(ctypes.byref(good), None, None, 4, 0, None, ctypes.byref(out))
    assert st == mc.MOE_ERR_INVALID_ARG and out.value is None
    assert "host_pool" in mc.moe_last_error()
