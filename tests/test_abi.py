"""The C-ABI library loads and exports every entry point its header declares.

CPU only: nothing here launches a kernel.  The argument checks exercised below
return before any CUDA call.
"""
import ctypes
import os
import re

import pytest

import paged_kv_cache_100_gb300 as pkv
from paged_kv_cache_100_gb300 import _lib
from paged_kv_cache_100_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for must in ("pa_decode", "pa_cache_write", "pa_block_copy", "pa_decode_workspace_bytes",
                 "pa_status_string", "pa_bm_create", "pa_bm_append_slot"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    assert sorted(_lib.SIGNATURES) == names, "binding signatures out of sync with the header"


def test_library_has_no_link_time_driver_dependency():
    # libcuda is reached through the runtime's driver entry points, so the
    # library also loads on machines without a GPU driver.
    maps = open("/proc/self/maps").read()
    assert _lib.LIB_PATH in maps or _lib.lib() is not None


def test_status_strings(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(5) == b"PA_ERR_WORKSPACE"
    assert lib.pa_status_string(99) == b"PA_ERR_UNKNOWN"
    assert lib.pa_version() >= 100


def test_partition_size_choice(lib):
    f = lib.pa_decode_partition_size
    # batch 64 x 32 KV heads up to 2064 tokens: plenty of CTAs with the longest partitions
    assert f(64, 32, 32, 129, 1) == 4096
    assert f(8, 32, 32, 129, 1) == 1024
    # one short sequence: no partition count reaches four CTAs per SM, smallest choice
    assert f(1, 8, 8, 4, 1) == 128
    # few sequences, long contexts: partitions shrink until there are enough CTAs
    p = f(2, 8, 8, 2048, 1)
    assert 128 <= p < 4096 and 2 * 8 * (-(-2048 * 16 // p)) >= 4 * 152
    # f32 counts query heads, bf16 KV heads
    assert f(8, 32, 4, 256, 0) >= f(8, 32, 4, 256, 1)
    assert f(-1, 4, 4, 4, 1) == -1 and f(1, 4, 4, 4, 9) == -1


def test_workspace_size_rules(lib):
    f = lib.pa_decode_workspace_bytes
    # one partition covers every sequence: nothing needed
    assert f(64, 32, 32, 128, 32, 16, 512, 1) == 0
    # 129 + 256 blocks -> 13 partitions of 512 tokens
    rows = 64 * 32 * 13
    need = f(64, 32, 32, 128, 129 + 256, 16, 512, 1)
    assert need >= rows * (128 * 4 + 8)
    bad = ctypes.c_size_t(-1).value
    assert f(1, 1, 1, 128, 4, 16, 100, 1) == bad          # not a multiple of 16
    assert f(1, 1, 1, 128, 4, 8, 0, 1) == bad             # block size must be 16
    assert f(1, 1, 1, 128, 4, 16, 32768, 1) == bad        # above the largest partition
    assert f(1, 1, 1, 128, 4, 16, 512, 5) == bad          # unknown dtype


def _decode_args(**over):
    a = dict(out=16, query=16, key_cache=16, value_cache=16, block_tables=16, context_lens=16,
             num_seqs=1, num_q_heads=4, num_kv_heads=4, head_dim=128, block_size=16,
             max_blocks=4, num_blocks=8, scale=0.1, dtype=1, partition_size=0, workspace=None,
             workspace_bytes=0, status=None, stream=None)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,expect", [
    (dict(block_size=8), _lib.PA_ERR_INVALID_ARG),
    (dict(num_q_heads=6, num_kv_heads=4), _lib.PA_ERR_INVALID_ARG),
    (dict(num_blocks=0), _lib.PA_ERR_INVALID_ARG),
    (dict(dtype=7), _lib.PA_ERR_INVALID_ARG),
    (dict(partition_size=24), _lib.PA_ERR_INVALID_ARG),
    (dict(out=None), _lib.PA_ERR_INVALID_ARG),
    (dict(key_cache=24), _lib.PA_ERR_INVALID_ARG),          # misaligned pool
    (dict(head_dim=96), _lib.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=68, num_kv_heads=2), _lib.PA_ERR_UNSUPPORTED),   # group 34
    (dict(max_blocks=100), _lib.PA_ERR_WORKSPACE),            # needs split-K scratch
    (dict(num_seqs=0, out=None), _lib.PA_OK),                 # nothing to do
])
def test_decode_argument_checks(lib, over, expect):
    assert lib.pa_decode(*_decode_args(**over)) == expect


def test_cache_write_and_block_copy_argument_checks(lib):
    cw = lib.pa_cache_write
    assert cw(16, 16, 16, 16, 16, 1, 8, 128, 8, 10, 1, None, None) == _lib.PA_ERR_INVALID_ARG
    assert cw(16, 16, 16, 16, 16, 1, 8, 4, 16, 10, 1, None, None) == _lib.PA_ERR_UNSUPPORTED
    assert cw(None, 16, 16, 16, 16, 1, 8, 128, 16, 10, 1, None, None) == _lib.PA_ERR_INVALID_ARG
    assert cw(None, None, None, None, None, 0, 8, 128, 16, 10, 1, None, None) == _lib.PA_OK
    bc = lib.pa_block_copy
    assert bc(16, 16, 16, 1, 8, 128, 16, 0, 1, None, None) == _lib.PA_ERR_INVALID_ARG
    assert bc(16, 16, None, 1, 8, 128, 16, 4, 1, None, None) == _lib.PA_ERR_INVALID_ARG
    assert bc(16, 16, 20, 1, 8, 128, 16, 4, 1, None, None) == _lib.PA_ERR_INVALID_ARG  # pairs not 8-byte aligned
    assert bc(None, None, None, 0, 8, 128, 16, 4, 1, None, None) == _lib.PA_OK


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 64, dtype=torch.bfloat16)
    kc = torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16)
    bt = torch.zeros(1, 1, dtype=torch.int32)
    cl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError):
        pkv.decode(q, kc, kc, bt, cl)


def test_shared_prefix_blocks_helper():
    import numpy as np
    t = np.array([[5, 6, 7, 9], [5, 6, 7, 10], [5, 6, 8, -1]], np.int32)
    assert pkv.shared_prefix_blocks(t) == 2
    assert pkv.shared_prefix_blocks(t[:2]) == 3
    assert pkv.shared_prefix_blocks(np.array([[1, -1], [1, -1]])) == 1


def test_shared_prefix_workspace_rules(lib):
    f = lib.pa_decode_shared_prefix_workspace_bytes
    bad = ctypes.c_size_t(-1).value
    assert f(128, 32, 8, 128, 129, 64, 0) > 0
    assert f(128, 32, 8, 128, 129, 200, 0) == bad         # prefix longer than the tables
    assert f(4, 6, 4, 128, 10, 2, 0) == bad               # heads not a multiple
