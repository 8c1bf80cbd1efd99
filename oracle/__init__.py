"""Oracle for paged decode attention, chunked prefill, cache write, block copy, swap
and the block manager.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product (``paged_kv_cache_100_gb300``) never imports it, and this package never
imports the product: the two share no code.

``pa_oracle.c`` is a plain fp64 C restatement of what the pages define (see the
header of that file for the page/section each function follows); this module
only compiles it with the host C compiler and marshals numpy arrays into it.
``block_manager_model`` is a plain-Python model of the host block manager.

Element types: float32 arrays are passed as float32; bfloat16 arrays are passed
as ``numpy.uint16`` arrays holding the raw 16-bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1
FP8_E4M3 = 2


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.pao_paged_decode.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                             i32, i32, i32, dbl, vp, i32, i32]
            lib.pao_paged_decode.restype = i32
            lib.pao_paged_decode_ex.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, i32,
                                                i32, i32, i32, i32, i32, i32, dbl, vp, i32, i32,
                                                i32]
            lib.pao_paged_decode_ex.restype = i32
            lib.pao_cache_write_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                                vp]
            lib.pao_cache_write_fp8.restype = i32
            lib.pao_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.pao_e4m3_value.restype = dbl
            lib.pao_e4m3_encode.argtypes = [ctypes.c_float]
            lib.pao_e4m3_encode.restype = ctypes.c_uint8
            lib.pao_cache_write.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32]
            lib.pao_cache_write.restype = i32
            lib.pao_block_copy.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                           ctypes.POINTER(ctypes.c_int)]
            lib.pao_block_copy.restype = i32
            lib.pao_paged_prefill.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, i32,
                                              i32, i32, i32, i32, i32, i32, dbl, i32, i32]
            lib.pao_paged_prefill.restype = i32
            lib.pao_max_threads.argtypes = []
            lib.pao_max_threads.restype = i32
            _lib = lib
        return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8:
        return FP8_E4M3
    raise TypeError(f"oracle expects float32, uint16 (bfloat16 bits) or uint8 (E4M3 codes), "
                    f"got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().pao_max_threads())


def paged_decode(query, key_cache, value_cache, block_tables, context_lens, scale,
                 sel=None, threads: int = 1, k_scales=None, v_scales=None,
                 window: int = 0) -> np.ndarray:
    """fp64 paged decode attention.

    query [B][Hq][D] (float32 or bfloat16 bits); key_cache/value_cache
    [NB][Hkv][BS][D] of the same type, or E4M3 codes (uint8) with per-KV-head
    ``k_scales`` / ``v_scales``; block_tables int32 [B][max_blocks]; context_lens
    int32 [B].  ``window`` > 0 attends only to the last ``window`` tokens.
    Returns float64 [B][Hq][D], or [n][D] for the (b, h) pairs of ``sel`` (an
    int array of shape [n, 2]).
    """
    lib = _load()
    query = np.ascontiguousarray(query)
    key_cache = np.ascontiguousarray(key_cache)
    value_cache = np.ascontiguousarray(value_cache)
    q_code = _dtype_code(query)
    kv_code = _dtype_code(key_cache)
    if _dtype_code(value_cache) != kv_code:
        raise TypeError("key_cache and value_cache must share one element type")
    if kv_code == FP8_E4M3:
        if k_scales is None or v_scales is None:
            raise ValueError("E4M3 pools need k_scales and v_scales")
    elif q_code != kv_code:
        raise TypeError("query and unquantised pools must share one element type")
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    if D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch between query and caches")
    if block_tables.ndim != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B][max_blocks] and context_lens [B]")
    ks = vs = None
    if kv_code == FP8_E4M3:
        ks = np.ascontiguousarray(k_scales, dtype=np.float32).reshape(Hkv)
        vs = np.ascontiguousarray(v_scales, dtype=np.float32).reshape(Hkv)
    if sel is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        sel_arr, n_sel = None, 0
    else:
        sel_arr = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
        n_sel = sel_arr.shape[0]
        out = np.zeros((n_sel, D), dtype=np.float64)
    rc = lib.pao_paged_decode_ex(out.ctypes.data, query.ctypes.data, q_code, key_cache.ctypes.data,
                                 value_cache.ctypes.data, kv_code,
                                 None if ks is None else ks.ctypes.data,
                                 None if vs is None else vs.ctypes.data,
                                 block_tables.ctypes.data, context_lens.ctypes.data, B, Hq, Hkv,
                                 D, BS, block_tables.shape[1], NB, float(scale),
                                 None if sel_arr is None else sel_arr.ctypes.data, n_sel,
                                 int(threads), int(window))
    if rc != 0:
        raise ValueError(f"oracle paged_decode failed with code {rc}")
    return out


def paged_prefill(query, key_cache, value_cache, block_tables, context_lens, query_start,
                  scale, threads: int = 1, k_scales=None, v_scales=None,
                  window: int = 0) -> np.ndarray:
    """fp64 chunked prefill over paged K/V (see ``pao_paged_prefill``).

    query [total_tokens][Hq][D]; sequence b's chunk is rows
    query_start[b] .. query_start[b+1]-1, the last T_b of its context_lens[b]
    positions (their K/V already in the pools).  Each row attends causally to
    the positions up to its own (the last ``window`` of them when ``window`` > 0).
    Returns float64 [total_tokens][Hq][D].
    """
    lib = _load()
    query = np.ascontiguousarray(query)
    key_cache = np.ascontiguousarray(key_cache)
    value_cache = np.ascontiguousarray(value_cache)
    q_code = _dtype_code(query)
    kv_code = _dtype_code(key_cache)
    if _dtype_code(value_cache) != kv_code:
        raise TypeError("key_cache and value_cache must share one element type")
    if kv_code == FP8_E4M3:
        if k_scales is None or v_scales is None:
            raise ValueError("E4M3 pools need k_scales and v_scales")
    elif q_code != kv_code:
        raise TypeError("query and unquantised pools must share one element type")
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    query_start = np.ascontiguousarray(query_start, dtype=np.int32)
    N, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    B = context_lens.shape[0]
    if D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch between query and caches")
    if block_tables.ndim != 2 or block_tables.shape[0] != B or query_start.shape != (B + 1,):
        raise ValueError("block_tables must be [B][max_blocks] and query_start [B + 1]")
    if int(query_start[-1]) != N:
        raise ValueError("query_start[B] must equal the number of query rows")
    ks = vs = None
    if kv_code == FP8_E4M3:
        ks = np.ascontiguousarray(k_scales, dtype=np.float32).reshape(Hkv)
        vs = np.ascontiguousarray(v_scales, dtype=np.float32).reshape(Hkv)
    out = np.zeros((N, Hq, D), dtype=np.float64)
    rc = lib.pao_paged_prefill(out.ctypes.data, query.ctypes.data, q_code, key_cache.ctypes.data,
                               value_cache.ctypes.data, kv_code,
                               None if ks is None else ks.ctypes.data,
                               None if vs is None else vs.ctypes.data,
                               block_tables.ctypes.data, context_lens.ctypes.data,
                               query_start.ctypes.data, B, Hq, Hkv, D, BS, block_tables.shape[1],
                               NB, float(scale), int(window), int(threads))
    if rc != 0:
        raise ValueError(f"oracle paged_prefill failed with code {rc}")
    return out


def e4m3_value(codes) -> np.ndarray:
    """float64 values of E4M3 codes (NaN for the two NaN codes)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.pao_e4m3_value(int(x)) for x in c.reshape(-1)]).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    """E4M3 codes of float32 values (nearest, ties to even, saturating at 448)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.pao_e4m3_encode(float(x)) for x in v.reshape(-1)],
                    dtype=np.uint8).reshape(v.shape)


def cache_write_fp8(key_cache, value_cache, key, value, slot_mapping, k_scales, v_scales):
    """In-place quantising cache write: bfloat16 rows [T][Hkv][D] into E4M3 pools."""
    lib = _load()
    for a in (key_cache, value_cache):
        if not a.flags.c_contiguous or a.dtype != np.uint8:
            raise ValueError("pools must be C-contiguous uint8 (written in place)")
    key = np.ascontiguousarray(key, dtype=np.uint16)
    value = np.ascontiguousarray(value, dtype=np.uint16)
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    NB, Hkv, BS, D = key_cache.shape
    T = slot_mapping.shape[0]
    if key.shape != (T, Hkv, D) or value.shape != (T, Hkv, D):
        raise ValueError("key/value must be [T][Hkv][D]")
    ks = np.ascontiguousarray(k_scales, dtype=np.float32).reshape(Hkv)
    vs = np.ascontiguousarray(v_scales, dtype=np.float32).reshape(Hkv)
    rc = lib.pao_cache_write_fp8(key_cache.ctypes.data, value_cache.ctypes.data, key.ctypes.data,
                                 value.ctypes.data, slot_mapping.ctypes.data, T, Hkv, D, BS, NB,
                                 ks.ctypes.data, vs.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle cache_write_fp8 failed with code {rc}")


def cache_write(key_cache, value_cache, key, value, slot_mapping) -> None:
    """In-place cache write into numpy pools [NB][Hkv][BS][D] from [T][Hkv][D] rows."""
    lib = _load()
    for a in (key_cache, value_cache):
        if not a.flags.c_contiguous:
            raise ValueError("pools must be C-contiguous (written in place)")
    key = np.ascontiguousarray(key)
    value = np.ascontiguousarray(value)
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    NB, Hkv, BS, D = key_cache.shape
    if key.dtype != key_cache.dtype or value.dtype != key_cache.dtype:
        raise TypeError("rows and pools must share one element type")
    T = slot_mapping.shape[0]
    if key.shape != (T, Hkv, D) or value.shape != (T, Hkv, D):
        raise ValueError("key/value must be [T][Hkv][D]")
    rc = lib.pao_cache_write(_ptr(key_cache), _ptr(value_cache), _ptr(key), _ptr(value),
                             _ptr(slot_mapping), T, Hkv, D, BS, NB, key_cache.itemsize)
    if rc != 0:
        raise ValueError(f"oracle cache_write failed with code {rc}")


def block_copy(key_cache, value_cache, pairs) -> bool:
    """In-place block copy; ``pairs`` is an int array [P][2] of (src, dst).

    Pairs are independent copies into fresh blocks (see ``pao_block_copy``):
    a pair with an index outside the pool, or whose dst is the src or dst of
    another pair (src != dst for both), is skipped.  Returns True when some
    pair was skipped."""
    lib = _load()
    for a in (key_cache, value_cache):
        if not a.flags.c_contiguous:
            raise ValueError("pools must be C-contiguous (written in place)")
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    NB, Hkv, BS, D = key_cache.shape
    skipped = ctypes.c_int(0)
    rc = lib.pao_block_copy(_ptr(key_cache), _ptr(value_cache), _ptr(pairs), pairs.shape[0],
                            Hkv, D, BS, NB, key_cache.itemsize, ctypes.byref(skipped))
    if rc != 0:
        raise ValueError(f"oracle block_copy failed with code {rc}")
    return bool(skipped.value)


def swap_out(key_cache, value_cache, block_ids) -> np.ndarray:
    """Preemption by swap ("PagedAttention por dentro", section "Evicción y
    preemption", strategy "swap"): the listed blocks copied out, in order, as
    staging[i] = (K tile of block_ids[i], V tile of block_ids[i]) over all KV
    heads; shape [n][2][Hkv][16][D] of the pools' element type."""
    ids = [int(b) for b in block_ids]
    NB, Hkv, BS, D = key_cache.shape
    staging = np.empty((len(ids), 2, Hkv, BS, D), dtype=key_cache.dtype)
    for i, b in enumerate(ids):
        if not 0 <= b < NB:
            raise IndexError(f"block id {b} outside the pool")
        staging[i, 0] = key_cache[b]
        staging[i, 1] = value_cache[b]
    return staging


def swap_in(key_cache, value_cache, block_ids, staging) -> None:
    """Inverse of ``swap_out``: staging[i] goes back into block block_ids[i] (in place)."""
    ids = [int(b) for b in block_ids]
    NB = key_cache.shape[0]
    if len(set(ids)) != len(ids):
        raise ValueError("swap-in block ids must be distinct")
    for i, b in enumerate(ids):
        if not 0 <= b < NB:
            raise IndexError(f"block id {b} outside the pool")
        key_cache[b] = staging[i, 0]
        value_cache[b] = staging[i, 1]
