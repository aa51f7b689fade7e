"""The C ABI library loads without a GPU and exports every function that
include/pa.h declares; host-only calls behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._libbuild().build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pa_pool_create", "pa_cache_append", "pa_decode", "pa_decode_split",
                 "pa_append_decode", "pa_copy_blocks", "pa_check", "pa_alloc_create"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_pool_bytes_give_the_pages_kv_sizes(lib):
    """2 * pool bytes of one block / 16 tokens = per-token per-layer KV bytes;
    times the layer count it reproduces the pages' 28 KiB (Qwen2.5-1.5B) and
    800 KiB (Llama 2 13B) per token."""
    f = lib.pa_pool_bytes
    f.restype = ctypes.c_size_t
    per_layer_qwen = 2 * f(1, 16, 2, 128, 1) // 16
    per_layer_l13 = 2 * f(1, 16, 40, 128, 0) // 16
    assert per_layer_qwen * 28 == 28 * 1024
    assert per_layer_l13 * 40 == 800 * 1024
    assert f(1, 8, 2, 128, 1) == 0 and f(1, 16, 2, 64, 1) == 0 and f(1, 16, 2, 128, 2) == 0


def test_host_side_validation_needs_no_gpu(lib):
    import paged_kv_cache_227_gb300 as pa
    h = ctypes.c_void_p()
    assert pa.lib.pa_pool_create(0, 16, 2, 128, 1, ctypes.byref(h)) == pa.PA_ERR_INVALID
    assert pa.lib.pa_pool_create(4, 32, 2, 128, 1, ctypes.byref(h)) == pa.PA_ERR_UNSUPPORTED
    assert pa.lib.pa_pool_create(4, 16, 2, 96, 1, ctypes.byref(h)) == pa.PA_ERR_UNSUPPORTED
    # 2^24 blocks x 8 heads x 16 rows = 2^31 token rows: past 32-bit row indices
    assert pa.lib.pa_pool_create(1 << 24, 16, 8, 128, 1, ctypes.byref(h)) == pa.PA_ERR_UNSUPPORTED
    assert pa.lib.pa_decode(None, None, None, 1, None, 1, 8, 1.0, None, 2, None) == pa.PA_ERR_INVALID
    assert pa.lib.pa_cache_append(None, None, None, None, 1, None) == pa.PA_ERR_INVALID
    assert pa.strerror(pa.PA_ERR_TIMEOUT).startswith("a bounded")
