"""ctypes loader for ``libpkv.so`` with the argument / return types of every
function that ``include/pkv.h`` declares."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
I32P = ctypes.POINTER(ctypes.c_int32)
SIZE = ctypes.c_size_t


class CacheDesc(ctypes.Structure):
    """``pkv_cache_desc``: geometry of one K or V page pool."""

    _fields_ = [
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("layout", ctypes.c_int32),
    ]


DESC_P = ctypes.POINTER(CacheDesc)

# name -> (restype, argtypes); mirrors include/pkv.h
SIGNATURES = {
    "pkv_append": (I32, [DESC_P, P, P, P, P, I32, P, P, I32, P, I32, P, P]),
    "pkv_decode_workspace_size": (SIZE, [I32, I32, I32, DESC_P]),
    "pkv_decode_attn": (I32, [DESC_P, P, P, P, P, P, P, I32, P, I32, I32, ctypes.c_float, P, P, P, SIZE, P, P]),
    "pkv_decode_attn_ex": (I32, [DESC_P, P, P, P, P, P, P, I32, P, I32, I32, ctypes.c_float, P, P, P, SIZE, P, P,
                                 ctypes.c_uint32]),
    "pkv_decode_attn_noalloc": (I32, [DESC_P, P, P, P, P, P, P, I32, P, I32, I32, ctypes.c_float, P, P, P, P]),
    "pkv_decode_bucket": (I32, [I32]),
    "pkv_decode_step_create": (I32, [DESC_P, I32, P, P, P, P, P, P, I32, P, I32, I32, ctypes.c_float, P, P, P, SIZE,
                                     P, ctypes.c_uint32, ctypes.POINTER(P)]),
    "pkv_decode_step_launch": (I32, [P, P]),
    "pkv_decode_step_destroy": (None, [P]),
    "pkv_prefill_workspace_size": (SIZE, [I32, I32, I32, DESC_P]),
    "pkv_prefill_attn": (I32, [DESC_P, P, P, P, P, P, P, I32, I32, I32, I32, ctypes.c_float, P, P, P, SIZE, P, P]),
    "pkv_mixed_workspace_size": (SIZE, [I32, I32, I32, I32, I32, I32, DESC_P]),
    "pkv_mixed_attn": (I32, [DESC_P, P, P, P, P, P, P, P, I32, P, I32, I32, I32, I32, I32, ctypes.c_float, P, P, P,
                             SIZE, P, P]),
    "pkv_pool_create": (P, [I32]),
    "pkv_pool_destroy": (None, [P]),
    "pkv_pool_alloc": (I32, [P, I32, I32P]),
    "pkv_pool_free": (I32, [P, I32P, I32]),
    "pkv_pool_num_free": (I32, [P]),
    "pkv_pool_shuffle": (I32, [P, ctypes.c_uint64]),
    "pkv_table_reserve": (I32, [P, I32P, I32, I32, I32, I32]),
    "pkv_table_release": (I32, [P, I32P, I32, I32, I32]),
    "pkv_validate_host": (I32, [DESC_P, I32P, I32, I32P, I32, I32, I32P]),
    "pkv_pool_bytes": (ctypes.c_uint64, [DESC_P]),
    "pkv_status_str": (ctypes.c_char_p, [I32]),
}


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Returns the loaded library, building it first if it is missing or older
    than its sources.  Raises if it cannot be built or loaded: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(_build.LIB_PATH):
                raise RuntimeError(f"CUDA library missing: {_build.LIB_PATH} (run __graft_entry__.build())")
            lib = ctypes.CDLL(_build.LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
