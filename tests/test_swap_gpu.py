"""GPU parity for swap: pa_swap_out / pa_swap_in bit-exact against the oracle, with
page-locked host staging (written and read by the kernel over the CPU-GPU link)
and with device staging, and a preempted sequence that decodes bit-identically
after its blocks were reused by another sequence and swapped back in."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_100_gb300.build import build
    build()
    import paged_kv_cache_100_gb300 as m
    return m


def _pools(dtype, NB=24, Hkv=4, D=128, seed=0):
    import torch
    rng = np.random.default_rng(seed)
    if dtype == "fp8":
        k = rng.integers(0, 256, (NB, Hkv, 16, D), dtype=np.uint8)
        v = rng.integers(0, 256, (NB, Hkv, 16, D), dtype=np.uint8)
        return k, v, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    x = rng.standard_normal((2, NB, Hkv, 16, D), dtype=np.float32)
    if dtype == "bf16":
        k, v = W.to_bf16_bits(x[0]), W.to_bf16_bits(x[1])
        return k, v, H.host_to_device(k, torch.bfloat16), H.host_to_device(v, torch.bfloat16)
    return x[0], x[1], torch.from_numpy(x[0]).cuda(), torch.from_numpy(x[1]).cuda()


def _bits(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32", "fp8"])
@pytest.mark.parametrize("where", ["host", "device"])
def test_swap_out_and_in_bit_exact(pkv, dtype, where):
    import torch
    k, v, kc, vc = _pools(dtype, seed=len(dtype))
    ids = np.array([7, 3, 19, 0, 23, 11], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    staging = None
    if where == "device":
        staging = torch.empty((len(ids), 2) + tuple(kc.shape[1:]), dtype=kc.dtype, device="cuda")
    staging = pkv.swap_out(kc, vc, torch.from_numpy(ids).cuda(), staging, status=status)
    torch.cuda.synchronize()
    assert staging.is_cuda == (where == "device")
    assert np.array_equal(_bits(staging), oracle.swap_out(k, v, ids))
    # back into other blocks (distinct ids; the rest of the pools unchanged)
    dst = np.array([1, 2, 4, 5, 6, 8], np.int32)
    pkv.swap_in(kc, vc, torch.from_numpy(dst).cuda(), staging, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    k2, v2 = k.copy(), v.copy()
    oracle.swap_in(k2, v2, dst, oracle.swap_out(k, v, ids))
    assert np.array_equal(_bits(kc), k2) and np.array_equal(_bits(vc), v2)


def test_out_of_range_ids_are_skipped_and_flagged(pkv):
    import torch
    k, v, kc, vc = _pools("bf16", NB=8, seed=3)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = torch.tensor([2, 8, -1, 5], dtype=torch.int32, device="cuda")
    staging = torch.zeros((4, 2) + tuple(kc.shape[1:]), dtype=kc.dtype, device="cuda")
    pkv.swap_out(kc, vc, ids, staging, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1                      # PA_DEV_BAD_BLOCK_ID
    got = _bits(staging)
    assert np.array_equal(got[[0, 3]], oracle.swap_out(k, v, [2, 5]))
    assert not got[[1, 2]].any()                        # skipped entries untouched
    status.zero_()
    pkv.swap_in(kc, vc, ids, staging, status=status)    # bad ids skipped on the way in too
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert np.array_equal(_bits(kc), k) and np.array_equal(_bits(vc), v)


def test_preempted_sequence_decodes_identically_after_swap(pkv):
    import torch
    NB, HKV, HQ, D = 40, 2, 8, 128
    bm = pkv.BlockManager(NB)
    lens = [70, 33, 120]
    for s, n in enumerate(lens):
        bm.alloc_seq(s, n)
    rng = np.random.default_rng(9)
    kc = H.host_to_device(W.to_bf16_bits(rng.standard_normal((NB, HKV, 16, D), dtype=np.float32)),
                          torch.bfloat16)
    vc = H.host_to_device(W.to_bf16_bits(rng.standard_normal((NB, HKV, 16, D), dtype=np.float32)),
                          torch.bfloat16)
    q = H.host_to_device(W.to_bf16_bits(rng.standard_normal((3, HQ, D), dtype=np.float32)),
                         torch.bfloat16)

    def decode():
        t, cl = bm.fill_tables([0, 1, 2], 10)
        out = pkv.decode(q, kc, vc, torch.from_numpy(t).cuda(), torch.from_numpy(cl).cuda(),
                         partition_size=32)
        torch.cuda.synchronize()
        return out

    before = decode()
    ids = bm.swap_out(2)                                # preempt seq 2
    staging = pkv.swap_out(kc, vc, torch.tensor(ids, dtype=torch.int32, device="cuda"))
    bm.alloc_seq(3, 16 * len(ids))                      # another request takes the blocks
    taken = bm.table(3)
    assert sorted(taken) == sorted(ids)
    junk = torch.full((len(taken), HKV, 16, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    idx = torch.tensor(taken, dtype=torch.long, device="cuda")
    kc[idx] = junk
    vc[idx] = junk
    new_ids = bm.swap_in(2)                             # seq 2 is scheduled again
    assert not set(new_ids) & set(taken)
    pkv.swap_in(kc, vc, torch.tensor(new_ids, dtype=torch.int32, device="cuda"), staging)
    after = decode()
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))
