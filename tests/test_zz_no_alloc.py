"""pa_decode_static_scratch: decode for callers that cannot allocate device memory.

Some callers cannot hand pa_decode a workspace: their device memory is reserved
up front by another allocator, or allocating (and the device synchronisation
that comes with it) is not acceptable where they run.  This entry point keeps
the split-K partials in a fixed library-owned device array instead.  The test
calls it through the C ABI and checks, on two calls in a row, that it gives the
same output as pa_decode with a workspace, within the bf16 tolerance used by
the other parity tests.  It lives in a file of its own that is collected last.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from paged_kv_cache_100_gb300.build import build
    build()
    import paged_kv_cache_100_gb300 as pkv
    return pkv


def _call_static(lib, out, q, kc, vc, bt, cl, wl, partition_size, status):
    import torch
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pa_decode_static_scratch(
        out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(),
        wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, bt.shape[1],
        wl.num_blocks, ctypes.c_float(wl.scale), 1, partition_size, status.data_ptr(), stream)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 4)])
def test_static_scratch_matches_workspace_decode_twice(built, hq, hkv):
    import torch
    pkv = built
    lib = pkv.lib()
    lens = [1, 100, 513, 1500, 3000]                  # several partitions of 256 tokens
    wl = W.custom_workload(len(lens), hq, hkv, 128, lens, dtype="bf16", seed=hq + hkv)
    partition_size = 256
    assert pkv.decode_workspace_bytes(wl.num_seqs, hq, hkv, 128, wl.max_blocks, partition_size) > 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        hv = W.host_values(wl, seed=100 + call)      # new inputs for each call
        q = H.host_to_device(hv.query, torch.bfloat16)
        kc = H.host_to_device(hv.key_cache, torch.bfloat16)
        vc = H.host_to_device(hv.value_cache, torch.bfloat16)
        bt = torch.from_numpy(wl.block_tables).cuda()
        cl = torch.from_numpy(wl.context_lens).cuda()
        want = pkv.decode(q, kc, vc, bt, cl, wl.scale, partition_size=partition_size)
        got = torch.full_like(want, float("nan"))
        rc = _call_static(lib, got, q, kc, vc, bt, cl, wl, partition_size, status)
        assert rc == 0, lib.pa_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        H.assert_close(H.as_f64(got), H.as_f64(want), "bf16", f"static scratch call {call}")


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
    rc = _call_static(lib, out, q, kc, kc, bt, cl, wl, 16, status)
    assert rc == pkv._lib.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert np.all(out.float().cpu().numpy() == 0)     # nothing was enqueued
