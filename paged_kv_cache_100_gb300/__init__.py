"""Paged KV-cache decode attention for GB300 (sm_103a).

A thin binding over the C ABI of ``include/pagedkv.h`` (library
``_build/libpagedkv.so``): every function here only turns torch tensors into
pointers and sizes and calls the library; all of the computation runs in the
library's CUDA kernels.  There is no CPU fallback.

    import paged_kv_cache_100_gb300 as pkv
    pkv.cache_write(key_cache, value_cache, k_new, v_new, slot_mapping)
    pkv.block_copy(key_cache, value_cache, cow_pairs)
    out = pkv.decode(query, key_cache, value_cache, block_tables, context_lens)

Layouts: pools [num_blocks][num_kv_heads][16][head_dim]; query/out
[num_seqs][num_q_heads][head_dim]; block_tables int32 [num_seqs][max_blocks];
context_lens int32 [num_seqs]; new rows [num_tokens][num_kv_heads][head_dim];
slot_mapping int64 [num_tokens]; copy pairs int32 [num_pairs][2].
"""
from __future__ import annotations

import ctypes
import math

from . import _lib
from ._lib import PagedKVError, check, lib  # noqa: F401

BLOCK_SIZE = 16

__all__ = ["prefill", "swap_out", "swap_in", "decode", "decode_fp8", "decode_sliding_window", "decode_shared_prefix", "decode_shared_prefix_fp8", "shared_prefix_blocks", "decode_workspace_bytes", "decode_partition_size",
           "cache_write", "cache_write_fp8", "block_copy", "launch_count", "BlockManager",
           "PagedKVError", "BLOCK_SIZE", "library_path"]


def library_path() -> str:
    return _lib.LIB_PATH


_TORCH = None


def _torch():
    global _TORCH
    if _TORCH is None:
        import torch
        _TORCH = torch
    return _TORCH


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return _lib.PA_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return _lib.PA_DTYPE_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return _lib.PA_DTYPE_FP8_E4M3
    raise TypeError(f"unsupported element type {t.dtype} (float32, bfloat16, or E4M3 codes as "
                    "uint8 / float8_e4m3fn)")


def _is_fp8(t) -> bool:
    torch = _torch()
    return t.dtype in (torch.uint8, torch.float8_e4m3fn)


def _dev(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream, t):
    """The given stream, else the current stream of tensor t's device."""
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return ctypes.c_void_p(raw(t.get_device()))
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _status_ptr(status):
    torch = _torch()
    if status is None:
        return None
    _dev(status, "status", torch.int32)
    return status.data_ptr()


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(lib().pa_launch_count())


def _code_of(dtype) -> int:
    name = str(dtype)
    if name in ("bf16", "torch.bfloat16"):
        return _lib.PA_DTYPE_BF16
    if name in ("fp8", "fp8_e4m3", "torch.uint8", "torch.float8_e4m3fn"):
        return _lib.PA_DTYPE_FP8_E4M3
    return _lib.PA_DTYPE_F32


def decode_partition_size(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq,
                          dtype="bf16") -> int:
    """Partition size (tokens) pa_decode picks when given partition_size=0."""
    code = _code_of(dtype)
    n = lib().pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq,
                                       code)
    if n < 0:
        raise ValueError("invalid arguments for pa_decode_partition_size")
    return int(n)


def decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                           partition_size=0, dtype="bf16") -> int:
    code = _code_of(dtype)
    n = lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                        max_blocks_per_seq, BLOCK_SIZE, partition_size, code)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid arguments for pa_decode_workspace_bytes")
    return int(n)


def decode(query, key_cache, value_cache, block_tables, context_lens, scale=None, *, out=None,
           partition_size=0, workspace=None, status=None, stream=None):
    """Paged decode attention (``pa_decode``); returns ``out``."""
    torch = _torch()
    B, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    if BS != BLOCK_SIZE or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("pools must be [num_blocks][num_kv_heads][16][head_dim] like query")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")
    code = _dtype_code(query)
    if key_cache.dtype != query.dtype or value_cache.dtype != query.dtype:
        raise TypeError("query and pools must share one element type")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(query)
    elif out.shape != query.shape or out.dtype != query.dtype:
        raise ValueError("out must match query")
    max_blocks = block_tables.shape[1]
    if workspace is None:
        # the library's scratch size for this call (0: none needed); a
        # caller's workspace is passed as given and sized by the library
        need = decode_workspace_bytes(B, Hq, Hkv, D, max_blocks, partition_size, query.dtype)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.nbytes
    rc = lib().pa_decode(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), B, Hq, Hkv, D, BLOCK_SIZE, max_blocks,
        NB, float(scale), code, int(partition_size), ws_ptr, ws_bytes, _status_ptr(status),
        _stream(stream, query))
    check(rc, "pa_decode")
    return out


def decode_shared_prefix(query, key_cache, value_cache, block_tables, context_lens,
                         num_prefix_blocks, scale=None, *, out=None, partition_size=0,
                         workspace=None, status=None, stream=None):
    """Decode for tables that all start with the same ``num_prefix_blocks`` blocks
    (``pa_decode_shared_prefix``); returns ``out``."""
    torch = _torch()
    B, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    if BS != BLOCK_SIZE or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("pools must be [num_blocks][num_kv_heads][16][head_dim] like query")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")
    code = _dtype_code(query)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(query)
    max_blocks = block_tables.shape[1]
    if workspace is None:
        need = lib().pa_decode_shared_prefix_workspace_bytes(B, Hq, Hkv, D, max_blocks,
                                                                int(num_prefix_blocks),
                                                                int(partition_size))
        if need == ctypes.c_size_t(-1).value:
            raise ValueError("invalid arguments for pa_decode_shared_prefix_workspace_bytes")
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=query.device)
    rc = lib().pa_decode_shared_prefix(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), B, Hq, Hkv, D, BLOCK_SIZE, max_blocks,
        NB, float(scale), code, int(num_prefix_blocks), int(partition_size),
        _dev(workspace, "workspace"), workspace.nbytes,
        _status_ptr(status), _stream(stream, query))
    check(rc, "pa_decode_shared_prefix")
    return out



def decode_shared_prefix_fp8(query, key_cache, value_cache, k_scales, v_scales, block_tables,
                             context_lens, num_prefix_blocks, scale=None, *, out=None,
                             partition_size=0, workspace=None, status=None, stream=None):
    """Shared-prefix decode over E4M3 pools (``pa_decode_shared_prefix_fp8``); returns
    ``out`` (bf16)."""
    torch = _torch()
    B, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    if BS != BLOCK_SIZE or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("pools must be [num_blocks][num_kv_heads][16][head_dim] like query")
    if not (_is_fp8(key_cache) and _is_fp8(value_cache)) or query.dtype != torch.bfloat16:
        raise TypeError("pa_decode_shared_prefix_fp8 takes E4M3 pools and a bfloat16 query")
    if k_scales.shape != (Hkv,) or v_scales.shape != (Hkv,):
        raise ValueError("k_scales / v_scales must be [num_kv_heads]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(query)
    max_blocks = block_tables.shape[1]
    if workspace is None:
        need = lib().pa_decode_shared_prefix_fp8_workspace_bytes(B, Hq, Hkv, D, max_blocks,
                                                                    int(num_prefix_blocks),
                                                                    int(partition_size))
        if need == ctypes.c_size_t(-1).value:
            raise ValueError("invalid arguments for pa_decode_shared_prefix_fp8_workspace_bytes")
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=query.device)
    rc = lib().pa_decode_shared_prefix_fp8(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(k_scales, "k_scales", torch.float32),
        _dev(v_scales, "v_scales", torch.float32),
        _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), B, Hq, Hkv, D, BLOCK_SIZE, max_blocks,
        NB, float(scale), int(num_prefix_blocks), int(partition_size),
        _dev(workspace, "workspace"), workspace.nbytes,
        _status_ptr(status), _stream(stream, query))
    check(rc, "pa_decode_shared_prefix_fp8")
    return out

def shared_prefix_blocks(block_tables) -> int:
    """Length (in blocks) of the physical prefix every row of host block tables shares."""
    import numpy as np
    t = np.asarray(block_tables)
    if t.shape[0] == 0:
        return 0
    same = np.all(t == t[0:1], axis=0) & (t[0] >= 0)
    n = int(np.argmin(same)) if not same.all() else t.shape[1]
    return n


def decode_fp8(query, key_cache, value_cache, k_scales, v_scales, block_tables, context_lens,
               scale=None, *, out=None, partition_size=0, workspace=None, status=None,
               stream=None):
    """Paged decode attention over E4M3 pools (``pa_decode_fp8``); returns ``out`` (bf16)."""
    torch = _torch()
    B, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    if BS != BLOCK_SIZE or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("pools must be [num_blocks][num_kv_heads][16][head_dim] like query")
    if not (_is_fp8(key_cache) and _is_fp8(value_cache)) or query.dtype != torch.bfloat16:
        raise TypeError("pa_decode_fp8 takes E4M3 pools and a bfloat16 query")
    if k_scales.shape != (Hkv,) or v_scales.shape != (Hkv,):
        raise ValueError("k_scales / v_scales must be [num_kv_heads]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(query)
    max_blocks = block_tables.shape[1]
    if workspace is None:
        # the library's scratch size for this call (0: none needed); a
        # caller's workspace is passed as given and sized by the library
        need = decode_workspace_bytes(B, Hq, Hkv, D, max_blocks, partition_size, "fp8")
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.nbytes
    rc = lib().pa_decode_fp8(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(k_scales, "k_scales", torch.float32),
        _dev(v_scales, "v_scales", torch.float32),
        _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), B, Hq, Hkv, D, BLOCK_SIZE, max_blocks,
        NB, float(scale), int(partition_size), ws_ptr, ws_bytes, _status_ptr(status),
        _stream(stream, query))
    check(rc, "pa_decode_fp8")
    return out


def decode_sliding_window(query, key_cache, value_cache, block_tables, context_lens, window,
                          scale=None, *, k_scales=None, v_scales=None, out=None,
                          partition_size=0, workspace=None, status=None, stream=None):
    """Decode over the last ``window`` positions of each context
    (``pa_decode_sliding_window``); bf16/fp32 pools, or E4M3 pools with
    ``k_scales``/``v_scales`` and a bf16 query.  Returns ``out``."""
    torch = _torch()
    B, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    if BS != BLOCK_SIZE or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("pools must be [num_blocks][num_kv_heads][16][head_dim] like query")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")
    if int(window) <= 0:
        raise ValueError("window must be positive")
    ks_ptr = vs_ptr = None
    if _is_fp8(key_cache):
        if not _is_fp8(value_cache) or query.dtype != torch.bfloat16:
            raise TypeError("E4M3 pools take a bfloat16 query")
        if k_scales is None or v_scales is None:
            raise ValueError("E4M3 pools need k_scales and v_scales")
        if k_scales.shape != (Hkv,) or v_scales.shape != (Hkv,):
            raise ValueError("k_scales / v_scales must be [num_kv_heads]")
        code = _lib.PA_DTYPE_FP8_E4M3
        ks_ptr = _dev(k_scales, "k_scales", torch.float32)
        vs_ptr = _dev(v_scales, "v_scales", torch.float32)
    else:
        code = _dtype_code(query)
        if key_cache.dtype != query.dtype or value_cache.dtype != query.dtype:
            raise TypeError("query and pools must share one element type")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(query)
    elif out.shape != query.shape or out.dtype != query.dtype:
        raise ValueError("out must match query")
    max_blocks = block_tables.shape[1]
    if workspace is None:
        need = lib().pa_decode_sliding_window_workspace_bytes(B, Hq, Hkv, D, max_blocks,
                                                              BLOCK_SIZE, int(window),
                                                              int(partition_size), code)
        if need == ctypes.c_size_t(-1).value:
            raise ValueError("invalid arguments for pa_decode_sliding_window_workspace_bytes")
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.nbytes
    rc = lib().pa_decode_sliding_window(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), ks_ptr, vs_ptr,
        _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), B, Hq, Hkv, D, BLOCK_SIZE, max_blocks,
        NB, float(scale), code, int(window), int(partition_size), ws_ptr, ws_bytes,
        _status_ptr(status), _stream(stream, query))
    check(rc, "pa_decode_sliding_window")
    return out


def cache_write_fp8(key_cache, value_cache, key, value, slot_mapping, k_scales, v_scales, *,
                    status=None, stream=None):
    """Quantise new bf16 K/V rows to E4M3 and scatter them into their slots."""
    torch = _torch()
    NB, Hkv, BS, D = key_cache.shape
    T = slot_mapping.shape[0]
    if key.shape != (T, Hkv, D) or value.shape != (T, Hkv, D):
        raise ValueError("key/value must be [num_tokens][num_kv_heads][head_dim]")
    if not (_is_fp8(key_cache) and _is_fp8(value_cache)):
        raise TypeError("pools must hold E4M3 codes")
    rc = lib().pa_cache_write_fp8(
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(key, "key", torch.bfloat16), _dev(value, "value", torch.bfloat16),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_scales, "k_scales", torch.float32),
        _dev(v_scales, "v_scales", torch.float32), T, Hkv, D, BS, NB, _status_ptr(status),
        _stream(stream, key_cache))
    check(rc, "pa_cache_write_fp8")


def cache_write(key_cache, value_cache, key, value, slot_mapping, *, status=None, stream=None):
    """Scatter new tokens' K/V rows into their slots (``pa_cache_write``)."""
    torch = _torch()
    NB, Hkv, BS, D = key_cache.shape
    T = slot_mapping.shape[0]
    if key.shape != (T, Hkv, D) or value.shape != (T, Hkv, D):
        raise ValueError("key/value must be [num_tokens][num_kv_heads][head_dim]")
    code = _dtype_code(key_cache)
    for t, n in ((value_cache, "value_cache"), (key, "key"), (value, "value")):
        if t.dtype != key_cache.dtype:
            raise TypeError(f"{n} must be {key_cache.dtype}")
    rc = lib().pa_cache_write(
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"), _dev(key, "key"),
        _dev(value, "value"), _dev(slot_mapping, "slot_mapping", torch.int64), T, Hkv, D, BS, NB,
        code, _status_ptr(status), _stream(stream, key_cache))
    check(rc, "pa_cache_write")


def block_copy(key_cache, value_cache, src_dst, *, status=None, stream=None):
    """Copy whole physical blocks (copy-on-write pairs) in both pools (``pa_block_copy``)."""
    torch = _torch()
    NB, Hkv, BS, D = key_cache.shape
    P = src_dst.shape[0]
    if src_dst.dim() != 2 or src_dst.shape[1] != 2:
        raise ValueError("src_dst must be [num_pairs][2]")
    rc = lib().pa_block_copy(
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(src_dst, "src_dst", torch.int32), P, Hkv, D, BS, NB, _dtype_code(key_cache),
        _status_ptr(status), _stream(stream, key_cache))
    check(rc, "pa_block_copy")


def prefill(query, key_cache, value_cache, block_tables, context_lens, query_start,
            max_query_len=None, scale=None, *, window=0, out=None, workspace=None, status=None,
            stream=None):
    """Chunked prefill over the paged pools (``pa_prefill``); returns ``out``.

    ``query`` [tokens][Hq][D] bf16 holds every sequence's chunk back to back,
    ``query_start`` (int32 [B+1]) where each begins; ``context_lens`` counts
    each context with its chunk.  ``max_query_len`` bounds the chunk lengths
    (read from ``query_start`` when omitted, which synchronises the stream)."""
    torch = _torch()
    N, Hq, D = query.shape
    NB, Hkv, BS, D2 = key_cache.shape
    B = context_lens.shape[0]
    if BS != BLOCK_SIZE or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("pools must be [num_blocks][num_kv_heads][16][head_dim] like query")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(query_start.shape) != (B + 1,):
        raise ValueError("block_tables must be [num_seqs][max_blocks], query_start [num_seqs + 1]")
    if query.dtype != torch.bfloat16 or key_cache.dtype != torch.bfloat16 or \
            value_cache.dtype != torch.bfloat16:
        raise TypeError("pa_prefill takes bfloat16 query and pools")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max().item()) if B else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(query)
    elif out.shape != query.shape or out.dtype != query.dtype:
        raise ValueError("out must match query")
    need = int(lib().pa_prefill_workspace_bytes())
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    rc = lib().pa_prefill(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32),
        _dev(query_start, "query_start", torch.int32), B, Hq, Hkv, D, BLOCK_SIZE,
        block_tables.shape[1], NB, N, int(max_query_len), float(scale), _lib.PA_DTYPE_BF16,
        int(window), _dev(workspace, "workspace"), workspace.nbytes,
        _status_ptr(status), _stream(stream, query))
    check(rc, "pa_prefill")
    return out


def _staging_ptr(t, nbytes):
    """Device-accessible staging: a CUDA tensor or a page-locked host tensor."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("staging must be a CUDA tensor or page-locked host memory")
    if not t.is_contiguous():
        raise ValueError("staging must be contiguous")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError("staging is too small")
    return t.data_ptr()


def _swap_geometry(key_cache, block_ids):
    torch = _torch()
    NB, Hkv, BS, D = key_cache.shape
    if block_ids.dim() != 1:
        raise ValueError("block_ids must be [num_ids]")
    code = _lib.PA_DTYPE_FP8_E4M3 if _is_fp8(key_cache) else _dtype_code(key_cache)
    n = block_ids.shape[0]
    nbytes = lib().pa_swap_bytes(n, Hkv, D, code)
    return NB, Hkv, BS, D, code, n, nbytes, _dev(block_ids, "block_ids", torch.int32)


def swap_out(key_cache, value_cache, block_ids, staging=None, *, status=None, stream=None):
    """Copy the listed blocks (both pools) into ``staging`` ``[n][2][Hkv][16][D]``
    (``pa_swap_out``).  By default the staging is new page-locked host memory,
    written by the kernel over the CPU-GPU link; returns it (complete once the
    stream reaches this point)."""
    torch = _torch()
    NB, Hkv, BS, D, code, n, nbytes, ids = _swap_geometry(key_cache, block_ids)
    if staging is None:
        staging = torch.empty((n, 2, Hkv, BS, D), dtype=key_cache.dtype, pin_memory=True)
    rc = lib().pa_swap_out(_dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"), ids,
                           n, _staging_ptr(staging, nbytes), Hkv, D, BS, NB, code,
                           _status_ptr(status), _stream(stream, key_cache))
    check(rc, "pa_swap_out")
    return staging


def swap_in(key_cache, value_cache, block_ids, staging, *, status=None, stream=None):
    """Copy ``staging`` back into the listed blocks (``pa_swap_in``); ids distinct."""
    NB, Hkv, BS, D, code, n, nbytes, ids = _swap_geometry(key_cache, block_ids)
    rc = lib().pa_swap_in(_dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"), ids,
                          n, _staging_ptr(staging, nbytes), Hkv, D, BS, NB, code,
                          _status_ptr(status), _stream(stream, key_cache))
    check(rc, "pa_swap_in")


class BlockManager:
    """Host block manager (``pa_bm_*``): pool, block tables, ref counts, copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE):
        self._h = lib().pa_bm_create(num_blocks, block_size)
        if not self._h:
            raise ValueError("bad pool geometry")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            lib().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc_seq(self, seq: int, num_tokens: int) -> None:
        check(lib().pa_bm_alloc_seq(self._h, seq, num_tokens), "pa_bm_alloc_seq")

    def fork(self, parent: int, child: int) -> None:
        check(lib().pa_bm_fork(self._h, parent, child), "pa_bm_fork")

    def append_slot(self, seq: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        check(lib().pa_bm_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                      ctypes.byref(dst)), "pa_bm_append_slot")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def make_private(self, seq: int, logical_block: int):
        src, dst = ctypes.c_int32(), ctypes.c_int32()
        check(lib().pa_bm_make_private(self._h, seq, logical_block, ctypes.byref(src),
                                       ctypes.byref(dst)), "pa_bm_make_private")
        return None if src.value < 0 else (src.value, dst.value)

    def free_seq(self, seq: int) -> None:
        check(lib().pa_bm_free_seq(self._h, seq), "pa_bm_free_seq")

    def num_free(self) -> int:
        return int(lib().pa_bm_num_free(self._h))

    def num_evictable(self) -> int:
        return int(lib().pa_bm_num_evictable(self._h))

    def alloc_seq_cached(self, seq: int, tokens) -> int:
        """New sequence reusing the prefix cache; returns the number of cached tokens."""
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int()
        check(lib().pa_bm_alloc_seq_cached(self._h, seq, t.ctypes.data, t.shape[0],
                                           ctypes.byref(n)), "pa_bm_alloc_seq_cached")
        return int(n.value)

    def register_prefix(self, seq: int, tokens) -> int:
        """Index the sequence's full blocks in the prefix cache; returns how many."""
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = lib().pa_bm_register_prefix(self._h, seq, t.ctypes.data, t.shape[0])
        if n < 0:
            raise KeyError(seq)
        return int(n)

    def trim_window(self, seq: int, window: int) -> int:
        """Release the blocks wholly before the last ``window`` tokens (their table
        entries become -1); returns how many were released."""
        if int(window) <= 0:
            raise ValueError("window must be positive")
        n = lib().pa_bm_trim_window(self._h, seq, int(window))
        if n < 0:
            raise KeyError(seq)
        return int(n)

    def swap_out(self, seq: int) -> list:
        """Release the sequence's blocks for a swap; returns them in staging order."""
        import numpy as np
        cap = max(1, len(self.table(seq)))
        ids = np.empty(cap, dtype=np.int32)
        n = ctypes.c_int()
        check(lib().pa_bm_swap_out(self._h, seq, ids.ctypes.data, cap, ctypes.byref(n)),
              "pa_bm_swap_out")
        return ids[:n.value].tolist()

    def swap_in(self, seq: int) -> list:
        """Fresh blocks for a swapped-out sequence, in staging order."""
        import numpy as np
        cap = max(1, len(self.table(seq)))
        ids = np.empty(cap, dtype=np.int32)
        n = ctypes.c_int()
        check(lib().pa_bm_swap_in(self._h, seq, ids.ctypes.data, cap, ctypes.byref(n)),
              "pa_bm_swap_in")
        return ids[:n.value].tolist()

    def num_tokens(self, seq: int) -> int:
        n = lib().pa_bm_num_tokens(self._h, seq)
        if n < 0:
            raise KeyError(seq)
        return int(n)

    def ref_count(self, block: int) -> int:
        return int(lib().pa_bm_ref_count(self._h, block))

    def table(self, seq: int) -> list:
        n = lib().pa_bm_table(self._h, seq, None, 0)
        if n < 0:
            raise KeyError(seq)
        buf = (ctypes.c_int32 * max(n, 1))()
        lib().pa_bm_table(self._h, seq, ctypes.cast(buf, ctypes.c_void_p), n)
        return list(buf[:n])

    def append_slots(self, seqs):
        """One decode step: returns (slots int64 [n], cow pairs int32 [k][2]) as numpy arrays."""
        import numpy as np
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        n = seqs.shape[0]
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int32)
        ncow, ndone = ctypes.c_int(), ctypes.c_int()
        rc = lib().pa_bm_append_slots(self._h, seqs.ctypes.data, n, slots.ctypes.data,
                                      pairs.ctypes.data, ctypes.byref(ncow), ctypes.byref(ndone))
        check(rc, f"pa_bm_append_slots (done {ndone.value} of {n})")
        return slots, pairs[:ncow.value].copy()

    def stats(self) -> dict:
        """Pool occupancy and internal fragmentation (``pa_bm_stats``)."""
        st = _lib.BmStats()
        check(lib().pa_bm_stats(self._h, ctypes.byref(st)), "pa_bm_stats")
        return {name: getattr(st, name) for name, _ in _lib.BmStats._fields_}

    def fill_tables(self, seqs, max_blocks: int):
        """Dense block tables [n][max_blocks] (-1 padded) and context lengths [n] (numpy)."""
        import numpy as np
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        n = seqs.shape[0]
        tables = np.empty((n, max_blocks), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        check(lib().pa_bm_fill_tables(self._h, seqs.ctypes.data, n, tables.ctypes.data,
                                      max_blocks, lens.ctypes.data), "pa_bm_fill_tables")
        return tables, lens
