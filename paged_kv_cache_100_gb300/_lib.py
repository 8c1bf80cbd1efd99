"""Loads ``_build/libpagedkv.so`` and declares the C ABI of ``include/pagedkv.h``.

There is no fallback: if the library is missing every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# PAGEDKV_LIBRARY may point at another build of the same library (e.g. a
# variant compiled with different tile parameters).
LIB_PATH = os.environ.get("PAGEDKV_LIBRARY") or os.path.join(HERE, "_build", "libpagedkv.so")

_lock = threading.Lock()
_lib = None

vp = ctypes.c_void_p
i32 = ctypes.c_int
i64 = ctypes.c_int64
u64 = ctypes.c_uint64
f32 = ctypes.c_float
sz = ctypes.c_size_t
ptr_i32 = ctypes.POINTER(ctypes.c_int32)
ptr_i64 = ctypes.POINTER(ctypes.c_int64)
ptr_int = ctypes.POINTER(ctypes.c_int)

# name -> (restype, argtypes); mirrors include/pagedkv.h
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [i32]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_version": (i32, []),
    "pa_launch_count": (u64, []),
    "pa_decode_partition_size": (i32, [i32, i32, i32, i32, i32]),
    "pa_decode_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32, i32]),
    "pa_decode": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, i32,
                        vp, sz, vp, vp]),
    "pa_decode_static_scratch": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                       f32, i32, i32, vp, vp]),
    "pa_decode_shared_prefix_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32]),
    "pa_decode_shared_prefix": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                      f32, i32, i32, i32, vp, sz, vp, vp]),
    "pa_decode_fp8": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                            i32, vp, sz, vp, vp]),
    "pa_decode_shared_prefix_fp8_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32]),
    "pa_decode_shared_prefix_fp8": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                          i32, i32, f32, i32, i32, vp, sz, vp, vp]),
    "pa_decode_sliding_window_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32, i32, i32,
                                                      i32]),
    "pa_decode_sliding_window": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                       i32, i32, f32, i32, i32, i32, vp, sz, vp, vp]),
    "pa_cache_write_fp8": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
    "pa_prefill_workspace_bytes": (sz, []),
    "pa_prefill": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                         f32, i32, i32, vp, sz, vp, vp]),
    "pa_swap_bytes": (sz, [i32, i32, i32, i32]),
    "pa_swap_out": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, vp, vp]),
    "pa_swap_in": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, vp, vp]),
    "pa_cache_write": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]),
    "pa_block_copy": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]),
    "pa_bm_create": (vp, [i32, i32]),
    "pa_bm_destroy": (None, [vp]),
    "pa_bm_alloc_seq": (i32, [vp, i32, i32]),
    "pa_bm_fork": (i32, [vp, i32, i32]),
    "pa_bm_append_slot": (i32, [vp, i32, ptr_i64, ptr_i32, ptr_i32]),
    "pa_bm_make_private": (i32, [vp, i32, i32, ptr_i32, ptr_i32]),
    "pa_bm_free_seq": (i32, [vp, i32]),
    "pa_bm_num_free": (i32, [vp]),
    "pa_bm_num_evictable": (i32, [vp]),
    "pa_bm_alloc_seq_cached": (i32, [vp, i32, vp, i32, ptr_int]),
    "pa_bm_register_prefix": (i32, [vp, i32, vp, i32]),
    "pa_bm_trim_window": (i32, [vp, i32, i32]),
    "pa_bm_swap_out": (i32, [vp, i32, vp, i32, ptr_int]),
    "pa_bm_swap_in": (i32, [vp, i32, vp, i32, ptr_int]),
    "pa_bm_num_tokens": (i32, [vp, i32]),
    "pa_bm_ref_count": (i32, [vp, i32]),
    "pa_bm_table": (i32, [vp, i32, vp, i32]),
    "pa_bm_append_slots": (i32, [vp, vp, i32, vp, vp, ptr_int, ptr_int]),
    "pa_bm_fill_tables": (i32, [vp, vp, i32, vp, i32, vp]),
    "pa_bm_stats": (i32, [vp, vp]),
}


class BmStats(ctypes.Structure):
    """pa_bm_stats_t"""
    _fields_ = [("num_blocks", ctypes.c_int64), ("free_blocks", ctypes.c_int64),
                ("evictable_blocks", ctypes.c_int64), ("used_blocks", ctypes.c_int64),
                ("shared_blocks", ctypes.c_int64), ("reserved_slots", ctypes.c_int64),
                ("filled_slots", ctypes.c_int64), ("logical_tokens", ctypes.c_int64),
                ("internal_fragmentation", ctypes.c_double)]

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_NO_BLOCKS = 4
PA_ERR_WORKSPACE = 5
PA_ERR_NOT_FOUND = 6

PA_DTYPE_F32 = 0
PA_DTYPE_BF16 = 1
PA_DTYPE_FP8_E4M3 = 2

PA_DEV_BAD_BLOCK_ID = 1
PA_DEV_BAD_CONTEXT_LEN = 2
PA_DEV_BAD_SLOT = 4
PA_DEV_BAD_COPY_PAIR = 8
PA_DEV_TIMEOUT = 16
PA_DEV_PREFIX_MISMATCH = 32
PA_DEV_BAD_QUERY_LEN = 64
PA_DEV_SMEM_ALIGN = 128
PA_DEV_RANGE = 256


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        name = lib().pa_status_string(status).decode()
        detail = lib().pa_last_error().decode() if status == PA_ERR_CUDA else ""
        super().__init__(f"{what}: {name}" + (f" ({detail})" if detail else ""))
        self.status = status


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"paged_kv_cache_100_gb300: CUDA library not built ({LIB_PATH} missing); "
                    "run paged_kv_cache_100_gb300.build.build() first")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedKVError(status, what)
