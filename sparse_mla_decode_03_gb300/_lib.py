"""ctypes loader of libsmla.so and the declarations of its C ABI (include/smla.h).

Loading fails loudly when the library has not been built: there is no fallback."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsmla.so")
# the same library built with SMLA_DEBUG (device-side bounds checks; see build.py)
DEBUG_LIB_PATH = os.path.join(_HERE, "libsmla_debug.so")

SMLA_OK = 0
SMLA_ERR_INVALID_ARG = -1
SMLA_ERR_UNSUPPORTED_SHAPE = -2
SMLA_ERR_WORKSPACE_TOO_SMALL = -3
SMLA_ERR_UNSUPPORTED_DEVICE = -4
SMLA_ERR_CUDA = -5
SMLA_ERR_TIMEOUT = -6
SMLA_ERR_INDEX_RANGE = -7
SMLA_ERR_RANGE = -8
SMLA_ERR_SCRATCH_TOO_SMALL = -9
SMLA_ERR_INTERNAL = -10

EXPORTED = (
    "smla_default_num_splits",
    "smla_decode_plan",
    "smla_workspace_size",
    "sparse_mla_decode",
    "sparse_mla_decode_split",
    "sparse_mla_combine",
    "sparse_mla_decode_noalloc",
    "sparse_mla_decode_simt",
    "smla_paged_workspace_size",
    "sparse_mla_decode_paged",
    "smla_status_string",
    "smla_device_status",
    "smla_test_inject_fault",
)


class SmlaParams(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("num_rows", ctypes.c_int64),
        ("kv_row_stride", ctypes.c_int64),
        ("softmax_scale", ctypes.c_float),
    ]


_lib = None
_debug_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _open(LIB_PATH)
    return _lib


def load_debug() -> ctypes.CDLL:
    """The SMLA_DEBUG build of the same C ABI (a separate library and device state)."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _open(DEBUG_LIB_PATH)
    return _debug_lib


def _open(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m sparse_mla_decode_03_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER(SmlaParams)
    lib.smla_default_num_splits.argtypes = [P, ctypes.POINTER(i32)]
    lib.smla_decode_plan.argtypes = [P, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.smla_workspace_size.argtypes = [P, i32, ctypes.POINTER(sz)]
    lib.sparse_mla_decode.argtypes = [vp, vp, vp, vp, vp, P, i32, vp, sz, vp]
    lib.sparse_mla_decode_split.argtypes = [vp, vp, vp, P, i32, vp, vp, vp]
    lib.sparse_mla_combine.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    lib.sparse_mla_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, P, i32, vp]
    lib.sparse_mla_decode_simt.argtypes = [vp, vp, vp, vp, vp, P, vp]
    lib.smla_paged_workspace_size.argtypes = [P, i32, ctypes.POINTER(sz)]
    lib.sparse_mla_decode_paged.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, P, i32, vp, sz, vp]
    lib.smla_status_string.argtypes = [ctypes.c_int]
    lib.smla_status_string.restype = ctypes.c_char_p
    lib.smla_device_status.argtypes = [ctypes.POINTER(i32), i32]
    lib.smla_test_inject_fault.argtypes = [i32]
    for name in EXPORTED:
        if name != "smla_status_string":
            getattr(lib, name).restype = ctypes.c_int
    return lib
