"""pa_decode_static_scratch: decode for callers that cannot allocate device memory.

Some callers cannot hand pa_decode a workspace: their device memory is reserved
up front by another allocator, or allocating (and the device synchronisation
that comes with it) is not acceptable where they run.  This entry point keeps
the split-K partials in a fixed library-owned device array instead.  The tests
call it through the C ABI, two calls in a row with different partition counts
(so the second call's partials sit at other offsets of the array than the
first's), and check each output against the fp64 oracle within the tolerance of
the other parity tests, and against pa_decode with a workspace.  This file is
collected last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from paged_kv_cache_100_gb300.build import build
    build()
    import paged_kv_cache_100_gb300 as pkv
    return pkv


def _call_static(lib, out, q, kc, vc, bt, cl, wl, partition_size, status, dtype_code):
    import torch
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pa_decode_static_scratch(
        None if out is None else out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
        bt.data_ptr(), cl.data_ptr(), wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
        16, bt.shape[1], wl.num_blocks, ctypes.c_float(wl.scale), dtype_code, partition_size,
        status.data_ptr(), stream)


# (query heads, KV heads, head_dim, dtype, partition sizes of the two calls):
# MHA and group-16 bf16, and the f32 kernel (one CTA per query head) with
# 16-token partitions so that its split path runs.
CASES = [(8, 8, 128, "bf16", (256, 64)), (32, 2, 128, "bf16", (512, 128)),
         (32, 4, 64, "bf16", (256, 1024)), (4, 4, 64, "f32", (16, 48))]


@pytest.mark.parametrize("hq,hkv,D,dtype,parts", CASES)
def test_static_scratch_matches_oracle_twice(built, hq, hkv, D, dtype, parts):
    import torch
    pkv = built
    lib = pkv.lib()
    lens = [1, 100, 513, 1500, 3000] if dtype == "bf16" else [1, 17, 33, 250, 700]
    wl = W.custom_workload(len(lens), hq, hkv, D, lens, dtype=dtype, seed=hq + hkv + D)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = 1 if dtype == "bf16" else 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, P in enumerate(parts):
        assert pkv.decode_workspace_bytes(wl.num_seqs, hq, hkv, D, wl.max_blocks, P, dtype) > 0
        hv = W.host_values(wl, seed=100 + call)      # new inputs for each call; unused slots NaN
        q = H.host_to_device(hv.query, tdt)
        kc = H.host_to_device(hv.key_cache, tdt)
        vc = H.host_to_device(hv.value_cache, tdt)
        bt = torch.from_numpy(wl.block_tables).cuda()
        cl = torch.from_numpy(wl.context_lens).cuda()
        got = torch.full_like(q, float("nan"))
        rc = _call_static(lib, got, q, kc, vc, bt, cl, wl, P, status, code)
        assert rc == 0, lib.pa_status_string(rc)
        want = pkv.decode(q, kc, vc, bt, cl, wl.scale, partition_size=P)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                                  wl.context_lens, wl.scale, threads=8)
        H.assert_close(H.as_f64(got), ref, dtype, f"static scratch call {call} against the oracle")
        H.assert_close(H.as_f64(got), H.as_f64(want), dtype, f"static scratch call {call} against pa_decode")


def test_static_scratch_rejects_requests_beyond_its_size(built):
    import torch
    pkv = built
    lib = pkv.lib()
    # 64 sequences x 64 heads x 64 partitions of 16 tokens need far more than the array
    wl = W.custom_workload(64, 64, 8, 128, [1024] * 64, dtype="bf16", seed=1)
    need = pkv.decode_workspace_bytes(64, 64, 8, 128, wl.max_blocks, 16)
    assert need > (32 << 20)
    q = torch.zeros(64, 64, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(wl.num_blocks, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    out = torch.zeros_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _call_static(lib, out, q, kc, kc, bt, cl, wl, 16, status, 1)
    assert rc == pkv._lib.PA_ERR_WORKSPACE
    # an invalid argument is reported as pa_decode reports it, even for a large request
    assert _call_static(lib, None, q, kc, kc, bt, cl, wl, 16, status, 1) == pkv._lib.PA_ERR_INVALID_ARG
    wl96 = W.custom_workload(64, 64, 8, 96, [1024] * 64, dtype="bf16", seed=1)
    assert _call_static(lib, out, q, kc, kc, bt, cl, wl96, 16, status, 1) == pkv._lib.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert np.all(out.float().cpu().numpy() == 0)     # nothing was enqueued
    assert int(status.item()) == 0
