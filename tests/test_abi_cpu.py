"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function declared in include/smla.h, and validates arguments before touching the
device."""
import ctypes
import os
import re

import pytest

from sparse_mla_decode_03_gb300 import _lib, make_params

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from sparse_mla_decode_03_gb300 import build
        build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"sparse_mla_decode", "sparse_mla_decode_split", "sparse_mla_combine"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(_lib.EXPORTED) <= names


def test_debug_build_exports_the_same_abi(lib):
    dbg = _lib.load_debug()
    for n in declared_functions():
        assert hasattr(dbg, n), f"{n} not exported by the SMLA_DEBUG build"
    assert "SMLA_ERR_INTERNAL" in dbg.smla_status_string(_lib.SMLA_ERR_INTERNAL).decode()


def test_status_strings(lib):
    for code in range(-10, 1):
        s = lib.smla_status_string(code).decode()
        assert s.startswith("SMLA")
    assert "unknown" in lib.smla_status_string(-99).decode()


def test_workspace_size_arithmetic(lib):
    p = make_params(32, 64, 2048, 1 << 20, 584)
    n = ctypes.c_size_t()
    assert lib.smla_workspace_size(ctypes.byref(p), 4, ctypes.byref(n)) == 0
    o = 32 * 64 * 4 * 448 * 4
    l = (32 * 64 * 4 * 4 + 255) // 256 * 256
    assert n.value == o + l


@pytest.mark.parametrize("field,value,code", [
    ("num_heads", 48, _lib.SMLA_ERR_UNSUPPORTED_SHAPE),
    ("num_heads", 256, _lib.SMLA_ERR_UNSUPPORTED_SHAPE),
    ("batch", 0, _lib.SMLA_ERR_INVALID_ARG),
    ("batch", 65536, _lib.SMLA_ERR_UNSUPPORTED_SHAPE),
    ("topk", 0, _lib.SMLA_ERR_INVALID_ARG),
    ("kv_row_stride", 580, _lib.SMLA_ERR_INVALID_ARG),
    ("kv_row_stride", 588, _lib.SMLA_ERR_INVALID_ARG),
    ("softmax_scale", 0.0, _lib.SMLA_ERR_INVALID_ARG),
    ("reserved", 1, _lib.SMLA_ERR_INVALID_ARG),
])
def test_param_validation(lib, field, value, code):
    p = make_params(2, 64, 128, 1000, 584)
    setattr(p, field, value)
    n = ctypes.c_size_t()
    assert lib.smla_workspace_size(ctypes.byref(p), 1, ctypes.byref(n)) == code


def test_split_count_bounds(lib):
    p = make_params(2, 64, 100, 1000, 584)       # 7 granules of 16
    n = ctypes.c_size_t()
    assert lib.smla_workspace_size(ctypes.byref(p), 7, ctypes.byref(n)) == 0
    assert lib.smla_workspace_size(ctypes.byref(p), 8, ctypes.byref(n)) == _lib.SMLA_ERR_INVALID_ARG
    assert lib.smla_workspace_size(ctypes.byref(p), -1, ctypes.byref(n)) == _lib.SMLA_ERR_INVALID_ARG


def test_null_pointers_rejected_before_any_launch(lib):
    p = make_params(2, 64, 128, 1000, 584)
    vp = ctypes.c_void_p
    st = lib.sparse_mla_decode(vp(0), vp(0), vp(0), vp(0), vp(0), ctypes.byref(p), 0, vp(0), 0,
                               vp(0))
    assert st == _lib.SMLA_ERR_INVALID_ARG
    st = lib.sparse_mla_combine(vp(0), vp(0), 1, 1, 1, vp(0), vp(0), vp(0))
    assert st == _lib.SMLA_ERR_INVALID_ARG


def test_paged_workspace_adds_the_translated_rows(lib):
    p = make_params(32, 64, 2048, 1 << 20, 584)
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.smla_workspace_size(ctypes.byref(p), 4, ctypes.byref(a)) == 0
    assert lib.smla_paged_workspace_size(ctypes.byref(p), 4, ctypes.byref(b)) == 0
    assert b.value == a.value + (32 * 2048 * 4 + 255) // 256 * 256


def test_paged_argument_checks(lib):
    p = make_params(2, 64, 128, 1000, 584)
    vp = ctypes.c_void_p
    args = (vp(16), vp(16), vp(16))
    # null block table, bad page size, bad table width: rejected before any launch
    assert lib.sparse_mla_decode_paged(vp(16), vp(16), vp(0), 4, 16, vp(16), vp(16), vp(16),
                                       ctypes.byref(p), 0, vp(256), 1 << 20, vp(0)) == \
        _lib.SMLA_ERR_INVALID_ARG
    assert lib.sparse_mla_decode_paged(vp(16), vp(16), vp(16), 4, 0, vp(16), vp(16), vp(16),
                                       ctypes.byref(p), 0, vp(256), 1 << 20, vp(0)) == \
        _lib.SMLA_ERR_INVALID_ARG
    assert lib.sparse_mla_decode_paged(vp(16), vp(16), vp(16), 0, 16, vp(16), vp(16), vp(16),
                                       ctypes.byref(p), 0, vp(256), 1 << 20, vp(0)) == \
        _lib.SMLA_ERR_INVALID_ARG
    del args
