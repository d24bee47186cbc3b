"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/pkv.h declares (no GPU needed, no compute calls)."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_210_gb300 as pkv
from paged_kv_cache_210_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for header in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if header.endswith(".h"):
            text = open(os.path.join(ROOT, "include", header)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pkv_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return ctypes.CDLL(lib_build.LIBRARY)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for required in ("pkv_pool_create", "pkv_append", "pkv_decode_attention",
                     "pkv_pool_destroy", "pkv_append_attend", "pkv_get_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    for name in declared_functions():
        assert name in pkv.EXPORTED, name


def test_status_strings(lib):
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(2).startswith(b"index out of range")


def test_create_rejects_bad_geometry_without_touching_the_device(lib):
    # geometry checks come before any CUDA call
    lib.pkv_pool_create.argtypes = [ctypes.POINTER(pkv.PoolConfig),
                                    ctypes.POINTER(ctypes.c_void_p)]
    h = ctypes.c_void_p()
    bad = [
        pkv.PoolConfig(16, 4096, 8, 32, 8, 64, 2048, 2, 0, 0),    # page size 8
        pkv.PoolConfig(16, 4096, 16, 32, 4, 64, 2048, 2, 0, 0),   # 4 kv heads
        pkv.PoolConfig(16, 4096, 16, 32, 8, 128, 2048, 2, 0, 0),  # head_dim 128
    ]
    for cfg in bad:
        assert lib.pkv_pool_create(ctypes.byref(cfg), ctypes.byref(h)) == pkv.PKV_ERR_UNSUPPORTED
    invalid = [
        pkv.PoolConfig(0, 4096, 16, 32, 8, 64, 2048, 2, 0, 0),    # no layers
        pkv.PoolConfig(16, 4096, 16, 32, 8, 64, 4096, 2, 0, 0),   # context past 2048
        pkv.PoolConfig(16, 4096, 16, 32, 8, 64, 2040, 2, 0, 0),   # not a page multiple
        pkv.PoolConfig(16, 4096, 16, 32, 8, 64, 2048, 0, 0, 0),   # no batch
        pkv.PoolConfig(16, 4096, 16, 32, 8, 64, 2048, 2, 129, 0), # too many splits
    ]
    for cfg in invalid:
        assert lib.pkv_pool_create(ctypes.byref(cfg), ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_pool_create(None, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG


def test_calls_on_a_null_handle_are_rejected(lib):
    P, i = ctypes.c_void_p, ctypes.c_int
    lib.pkv_append.argtypes = [P, i, P, P, P, P, P, P, i, P]
    lib.pkv_decode_attention.argtypes = [P, i, P, P, P, P, P, P, i, i, P]
    lib.pkv_get_error.argtypes = [P, P]
    lib.pkv_pool_destroy.argtypes = [P]
    assert lib.pkv_append(None, 0, 16, 16, 16, 16, 16, 16, 1, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention(None, 0, 16, 16, 16, 16, 16, 16, 1, 0, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_get_error(None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_pool_destroy(None) == pkv.PKV_OK


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        pkv.load(str(tmp_path / "libpkv.so"))
