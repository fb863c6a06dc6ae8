"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and its host-only logic (Eq. 21.2 bytes, argument validation that fails
before any CUDA call) behaves."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import paged_kv_cache_kvc_gb300 as k
    if not os.path.exists(k.LIB_PATH):
        from paged_kv_cache_kvc_gb300 import build
        build.build()
    return k.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    return sorted(set(re.findall(r"KVC_API\s+[\w\s\*]+?\b(kvc_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    import paged_kv_cache_kvc_gb300 as k
    assert sorted(k.EXPORTS) == names


def test_kvc_bytes_matches_oracle_on_page_values(lib):
    import oracle
    import paged_kv_cache_kvc_gb300 as k
    cases = [(1, 1, 1, 3, 2, 2), (1, 1, 1, 4, 2, 2), (32, 1, 8, 8192, 128, 2), (2, 1, 4, 8, 8, 2),
             (32, 1, 8, 1, 128, 2), (32, 8, 8, 32768, 128, 2), (-1, 1, 1, 1, 1, 1), (2**20, 2**20, 2**20, 2**20, 1, 1)]
    for c in cases:
        assert k.kvc_bytes(*c) == oracle.kv_bytes(*c)
    assert k.kvc_bytes(1, 1, 1, 3, 2, 2) == 24 and k.kvc_bytes(32, 1, 8, 1, 128, 2) == 131072


def test_status_strings(lib):
    import paged_kv_cache_kvc_gb300 as k
    for s in range(10):
        assert k.kvc_status_str(s)
    assert k.kvc_status_str(0) == "ok"


def test_pool_create_rejects_bad_shapes_before_cuda(lib):
    import paged_kv_cache_kvc_gb300 as k
    out = ctypes.c_void_p(1)
    for args in [(0, 16, 1, 8, 128, 0), (10, 0, 1, 8, 128, 0), (10, 16, 1, 8, 96, 0), (10, 16, 1, 8, 64, 1),
                 (10, 16, 1, 8, 256, 0), (10, 16, 1, 8, 256, 1), (10, 16, 1, 8, 64, 2), (10, 129, 1, 8, 128, 0),
                 (10, 16, 0, 8, 128, 0), (10, 16, 1, 8, 128, 7), (2**40, 16, 1, 8, 128, 0)]:
        assert lib.kvc_pool_create(*args, ctypes.byref(out)) == k.KVC_ERR_ARG
        assert out.value is None


def test_null_pool_calls_are_argument_errors(lib):
    import paged_kv_cache_kvc_gb300 as k
    assert lib.kvc_pool_info(None, None) == k.KVC_ERR_ARG
    assert lib.kvc_decode_attn(None, 0, None, 8, None, 1, None, 1, None, None, 1.0, None) == k.KVC_ERR_ARG
    assert lib.kvc_append(None, 0, None, 1, None, 1, None, None, None) == k.KVC_ERR_ARG
    assert lib.kvc_pool_sync_status(None, None) == k.KVC_ERR_ARG
    lib.kvc_pool_destroy(None)


def test_product_path_fails_loudly_without_library(tmp_path):
    import importlib
    import paged_kv_cache_kvc_gb300 as k
    saved = k._lib
    try:
        k._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            k.load(str(tmp_path / "missing.so"))
    finally:
        k._lib = saved
        importlib.reload(k) if saved is None else None
