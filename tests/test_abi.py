"""The C-ABI library builds for sm_103a, loads, and exports every symbol the
header declares; argument checks that need no GPU return their error codes."""
import ctypes as C
import os
import re

import pytest

from swiftkv_prefill_skipping_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swiftkv.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swiftkv_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_cache_count_and_errors_without_gpu():
    lib = B.lib()
    assert lib.swiftkv_cache_count(32, 16, 1) == 32
    assert lib.swiftkv_cache_count(32, 16, 2) == 24
    assert lib.swiftkv_cache_count(32, 16, 4) == 20
    assert lib.swiftkv_cache_count(48, 24, 4) == 30
    assert lib.swiftkv_cache_count(32, 32, 1) == 32
    assert lib.swiftkv_cache_count(32, 0, 1) == -2
    assert lib.swiftkv_cache_count(32, 33, 1) == -2
    assert lib.swiftkv_cache_count(32, 16, 3) == -3
    assert lib.swiftkv_cache_count(32, 16, 0) == -3
    assert b"group" in lib.swiftkv_last_error()


def test_model_create_rejects_bad_config_before_touching_the_gpu():
    lib = B.lib()
    h = C.c_void_p()
    cfg = B.ModelConfig(4, 256, 4, 2, 96, 688, 1024, 0, 10000.0, 1e-5)   # d_head 96 unsupported
    assert lib.swiftkv_model_create(C.byref(cfg), 2, 1, C.byref(h)) == -9
    cfg = B.ModelConfig(4, 256, 4, 3, 64, 688, 1024, 0, 10000.0, 1e-5)   # 4 % 3 != 0
    assert lib.swiftkv_model_create(C.byref(cfg), 2, 1, C.byref(h)) == -9
    cfg = B.ModelConfig(4, 256, 4, 2, 64, 688, 1024, 0, 10000.0, 1e-5)
    assert lib.swiftkv_model_create(C.byref(cfg), 5, 1, C.byref(h)) == -2
    assert lib.swiftkv_model_create(C.byref(cfg), 1, 2, C.byref(h)) == -3
    assert h.value is None
    assert lib.swiftkv_prefill(None, None, None, 1, 1, 1, None, None, None) == -1
    assert lib.swiftkv_status(None, 0) == -1
    lib.swiftkv_free(None)


def test_no_cpu_fallback_in_product_path():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "swiftkv_prefill_skipping_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn


def test_timeout_selftest_argument_checks_without_gpu():
    """Limits outside [1 us, 100 ms] and a NULL status are refused before anything launches."""
    lib = B.lib()
    fake = C.c_void_p(256)   # never dereferenced: the arguments are rejected first
    for bad in (0, 999, 100_000_001):
        assert lib.swiftkv_selftest_wait_timeout(fake, None, bad, None) == -1
    assert lib.swiftkv_selftest_wait_timeout(None, None, 1_000_000, None) == -1

