"""GPU: the f16 staging of some paths is flagged, not silent, outside f16's range.

pa_prefill (and the tensor-core prefix of pa_decode_shared_prefix) convert V to
f16 for P.V; the FP8 decode consumers round the query to f16.  f16's largest
finite value is 65504, and bf16 has no value between 65280 and 65536, so an
element of magnitude 65536 or more cannot be staged exactly: the call must
raise PA_DEV_RANGE.  Elements below that (40000 here) must not."""
import numpy as np
import pytest

import workloads as W
from tests import helpers as H
from tests.test_prefill_gpu import _case, _run
from tests.test_shared_prefix_gpu import _shared_workload

pytestmark = pytest.mark.gpu

BIG = 1.0e5          # beyond f16
LARGE = 40000.0      # within f16


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_100_gb300.build import build
    build()
    import paged_kv_cache_100_gb300 as m
    return m


def _set_context_v(wl, hv, b, pos, value):
    phys = int(wl.block_tables[b, pos // 16])
    hv.value_cache[phys, :, pos % 16, 3] = W.to_bf16_bits(np.float32([value]))[0]


@pytest.mark.parametrize("value,flagged", [(BIG, True), (-BIG, True), (np.inf, True), (LARGE, False)])
def test_prefill_v_beyond_f16_is_flagged(pkv, value, flagged):
    wl, hv, q, qs, tables, lens = _case(8, 2, [(0, 40), (100, 130)], seed=71)
    _set_context_v(wl, hv, 1, 57, value)             # a cached position every chunk row attends to
    _, st = _run(pkv, wl, hv, q, qs, tables, lens)
    assert bool(st & pkv._lib.PA_DEV_RANGE) == flagged
    assert st & ~pkv._lib.PA_DEV_RANGE == 0


@pytest.mark.parametrize("value,flagged", [(BIG, True), (LARGE, False)])
def test_shared_prefix_v_beyond_f16_is_flagged(pkv, value, flagged):
    import torch
    wl = _shared_workload(6, 32, 8, 128, 8, [0, 3, 17, 40, 100, 5], seed=72)
    hv = W.host_values(wl)
    _set_context_v(wl, hv, 0, 20, value)             # a prefix position (block 1 of 8)
    kc = H.host_to_device(hv.key_cache, torch.bfloat16)
    vc = H.host_to_device(hv.value_cache, torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.decode_shared_prefix(H.host_to_device(hv.query, torch.bfloat16), kc, vc,
                             torch.from_numpy(wl.block_tables).cuda(),
                             torch.from_numpy(wl.context_lens).cuda(), 8, wl.scale, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert bool(st & pkv._lib.PA_DEV_RANGE) == flagged
    assert st & ~pkv._lib.PA_DEV_RANGE == 0


# (8, 8) with 16384-token partitions takes the CUDA-core MHA consumer (spans of
# more than 64 blocks), the others the tensor-core consumer
@pytest.mark.parametrize("hq,hkv,lens,P", [(8, 8, [300, 40], 0), (8, 8, [2000, 3], 16384),
                                           (16, 2, [300, 40], 0)])
@pytest.mark.parametrize("value,flagged", [(BIG, True), (-np.inf, True), (LARGE, False)])
def test_fp8_query_beyond_f16_is_flagged(pkv, hq, hkv, lens, P, value, flagged):
    import torch
    wl = W.custom_workload(len(lens), hq, hkv, 128, lens, dtype="bf16", seed=73)
    hv = W.fp8_host_values(wl)
    hv.query[1, hq - 1, 77] = W.to_bf16_bits(np.float32([value]))[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pkv.decode_fp8(H.host_to_device(hv.query, torch.bfloat16), dev(hv.key_cache),
                   dev(hv.value_cache), dev(hv.k_scales), dev(hv.v_scales),
                   dev(wl.block_tables), dev(wl.context_lens), wl.scale, partition_size=P,
                   status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert bool(st & pkv._lib.PA_DEV_RANGE) == flagged
    assert st & ~pkv._lib.PA_DEV_RANGE == 0
