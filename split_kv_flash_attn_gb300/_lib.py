"""ctypes binding of libsplitkv.so (the C ABI in include/splitkv.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  If the shared library has not been built this module
raises at import time -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsplitkv.so")

SKV_OK = 0
STATUS = {0: "SKV_OK", 1: "SKV_EINVAL", 2: "SKV_EUNSUPPORTED", 3: "SKV_ENOTPINNED", 4: "SKV_ENOMEM",
          5: "SKV_ECAPTURE", 6: "SKV_ECUDA", 7: "SKV_ETIMEOUT", 8: "SKV_EDEVICE"}
F16, Q8_0, Q4_0 = 0, 1, 2

# Every entry point that include/splitkv.h declares.
EXPORTS = [
    "skv_create", "skv_destroy", "skv_last_error", "skv_status_string", "skv_reserve", "skv_scratch_info",
    "skv_sm_count", "skv_status", "skv_set_profile_events", "skv_plan_splits", "skv_plan_prefill_splits", "skv_attn_partial", "skv_attn_combine", "skv_attn_window_tail",
    "skv_kv_dequant_q8_0", "skv_kv_dequant_q4_0", "skv_gather_rows", "skv_kv_append",
    "skv_attn_paged", "skv_bcache_create", "skv_bcache_destroy", "skv_bcache_reset", "skv_bcache_resolve",
    "skv_bcache_append", "skv_bcache_attn", "skv_bcache_stats", "skv_bcache_check", "skv_bcache_pool",
    "skv_bcache_create_ring", "skv_bcache_ring_restore", "skv_bcache_ring_attn",
    "skv_attn_partial_static", "skv_plan_window", "skv_plan_tail_tile", "skv_selftest_wait_timeout",
]


class SkvBcacheCounters(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("lookups", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("overflow", ctypes.c_uint64), ("last_misses", ctypes.c_int64),
                ("last_overflow", ctypes.c_int64)]


class SkvShape(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int32), ("nq", ctypes.c_int32), ("H", ctypes.c_int32), ("Hk", ctypes.c_int32),
                ("D", ctypes.c_int32), ("scale", ctypes.c_float), ("k_type", ctypes.c_int32),
                ("v_type", ctypes.c_int32), ("k_row_bytes", ctypes.c_int64), ("v_row_bytes", ctypes.c_int64)]


def _declare(lib):
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    SH = ctypes.POINTER(SkvShape)
    sig = {
        "skv_create": ([ctypes.c_int, ctypes.POINTER(P)], ctypes.c_int),
        "skv_destroy": ([P], ctypes.c_int),
        "skv_last_error": ([P], ctypes.c_char_p),
        "skv_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "skv_reserve": ([P, SZ, SZ, I32], ctypes.c_int),
        "skv_scratch_info": ([P, ctypes.POINTER(SZ), ctypes.POINTER(SZ), ctypes.POINTER(I32)], ctypes.c_int),
        "skv_sm_count": ([P, ctypes.POINTER(I32)], ctypes.c_int),
        "skv_set_profile_events": ([P, P, P], ctypes.c_int),
        "skv_status": ([P, ctypes.POINTER(I32)], ctypes.c_int),
        "skv_plan_splits": ([I64, I64, I32, I32, I32, I64, ctypes.POINTER(I64), ctypes.POINTER(I32)], ctypes.c_int),
        "skv_plan_prefill_splits": ([SH, I64, I32, I32, ctypes.POINTER(I64), ctypes.POINTER(I32), ctypes.POINTER(I64)],
                                    ctypes.c_int),
        "skv_attn_partial": ([P, SH, P, P, P, P, I64, P, I64, P, I64, I32, I64, I64, P, P, P], ctypes.c_int),
        "skv_attn_combine": ([P, I32, P, P, I64, I32, P, P, P], ctypes.c_int),
        "skv_attn_window_tail": ([P, SH, P, P, P, I64, P, P, I64, I64, P, I64, P, P, P, P], ctypes.c_int),
        "skv_kv_dequant_q8_0": ([P, P, I64, P, P], ctypes.c_int),
        "skv_kv_dequant_q4_0": ([P, P, I64, P, P], ctypes.c_int),
        "skv_gather_rows": ([P, P, I64, P, I64, P, P], ctypes.c_int),
        "skv_selftest_wait_timeout": ([P, I64, P], ctypes.c_int),
        "skv_kv_append": ([P, I32, I32, I32, I64, P, P, I32, P, I64, P, I64, P], ctypes.c_int),
        "skv_bcache_append": ([P, P, P, P, I32, P], ctypes.c_int),
        "skv_bcache_create_ring": ([P, I64, I32, I32, I32, I32, I32, P, P, ctypes.POINTER(P)], ctypes.c_int),
        "skv_bcache_ring_restore": ([P, I64, P], ctypes.c_int),
        "skv_bcache_ring_attn": ([P, SH, P, I64, I64, P, P, P], ctypes.c_int),
        "skv_plan_window": ([I64, I64, I64, I64, I64, I32, ctypes.POINTER(I64)], ctypes.c_int),
        "skv_plan_tail_tile": ([I64, I64, I32, I64, I64, I32, ctypes.POINTER(I64), ctypes.POINTER(I32)],
                               ctypes.c_int),
        "skv_attn_paged": ([P, SH, P, P, P, I32, P, I32, P, P, P], ctypes.c_int),
        "skv_attn_partial_static": ([SH, P, P, P, P, I64, P, I64, P, I64, I32, I64, I64, P, P, P], ctypes.c_int),
        "skv_bcache_create": ([P, I64, I32, I32, I32, I32, I64, P, P, ctypes.POINTER(P)], ctypes.c_int),
        "skv_bcache_destroy": ([P], ctypes.c_int),
        "skv_bcache_reset": ([P, P], ctypes.c_int),
        "skv_bcache_resolve": ([P, P, I32, I32, P, P], ctypes.c_int),
        "skv_bcache_attn": ([P, SH, P, P, I32, P, P, P], ctypes.c_int),
        "skv_bcache_stats": ([P, ctypes.POINTER(SkvBcacheCounters)], ctypes.c_int),
        "skv_bcache_check": ([P, ctypes.POINTER(I32)], ctypes.c_int),
        "skv_bcache_pool": ([P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(I64), ctypes.POINTER(P)],
                            ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res


def load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"libsplitkv.so is not built ({path}); run __graft_entry__.build() "
                          "or python split_kv_flash_attn_gb300/build.py")
    lib = ctypes.CDLL(path)
    _declare(lib)
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load()
    return _lib
