"""GPU parity for FP8 (E4M3) pools: pa_cache_write_fp8 (bit-exact), pa_decode_fp8
(within the bf16-output tolerance) and pa_block_copy on 1-byte elements."""
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


def _dev_u8(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bf16(a):
    import torch
    return H.host_to_device(a, torch.bfloat16)


def _decode(pkv, wl, hv, lens=None, partition_size=0):
    import torch
    lens = wl.context_lens if lens is None else lens
    out = pkv.decode_fp8(_bf16(hv.query), _dev_u8(hv.key_cache), _dev_u8(hv.value_cache),
                         _dev_u8(hv.k_scales), _dev_u8(hv.v_scales),
                         torch.from_numpy(wl.block_tables).cuda(),
                         torch.from_numpy(np.asarray(lens, np.int32)).cuda(), wl.scale,
                         partition_size=partition_size)
    torch.cuda.synchronize()
    return out


def _oracle(wl, hv, lens=None):
    lens = wl.context_lens if lens is None else lens
    return oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                               np.asarray(lens, np.int32), wl.scale, threads=4,
                               k_scales=hv.k_scales, v_scales=hv.v_scales)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (12, 4), (6, 3), (16, 8)])
@pytest.mark.parametrize("partition_size", [0, 64, 16384])
def test_decode_fp8_matches_oracle(pkv, hq, hkv, partition_size):
    lens = [1, 15, 16, 17, 100, 513, 1100]
    wl = W.custom_workload(len(lens), hq, hkv, 128, lens, dtype="bf16", seed=hq * 3 + hkv)
    hv = W.fp8_host_values(wl)                       # unused slots hold the NaN code
    got = H.as_f64(_decode(pkv, wl, hv, partition_size=partition_size))
    H.assert_close(got, _oracle(wl, hv), "bf16", f"fp8 {hq}/{hkv} P={partition_size}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2)])
@pytest.mark.parametrize("partition_size", [0, 16384])
def test_decode_fp8_empty_and_one_token_contexts(pkv, hq, hkv, partition_size):
    """An empty context gives zeros; a one-token context gives that token's value
    (code times its head's scale, rounded to bf16), on the tensor-core and the
    CUDA-core MHA consumers alike."""
    lens = [0, 1, 40, 0, 1]
    wl = W.custom_workload(len(lens), hq, hkv, 128, lens, dtype="bf16", seed=hq + hkv + 5)
    hv = W.fp8_host_values(wl)
    got = H.as_f64(_decode(pkv, wl, hv, partition_size=partition_size))
    assert np.all(got[0] == 0) and np.all(got[3] == 0)
    H.assert_close(got, _oracle(wl, hv), "bf16", f"fp8 short contexts {hq}/{hkv} P={partition_size}")


def test_cache_write_fp8_bit_exact_including_saturation_and_tiny_values(pkv):
    import torch
    wl = W.custom_workload(6, 8, 4, 128, [0, 15, 16, 31, 300, 7], dtype="bf16", seed=2)
    hv = W.fp8_host_values(wl)
    kx = W.bf16_bits_to_f32(hv.key_new).copy()
    kx[0, 0, :8] *= 1e3                               # saturates at +-448
    kx[1, 1, :8] *= 1e-4                              # subnormal codes
    kx[2, 2, :4] = [0.0, -0.0, 1e-30, -1e-30]         # zeros of both signs
    kn = W.to_bf16_bits(kx)
    slots = wl.slot_mapping.copy()
    slots[5] = -1                                     # padding: no write
    kc, vc = _dev_u8(hv.key_cache), _dev_u8(hv.value_cache)
    pkv.cache_write_fp8(kc, vc, _bf16(kn), _bf16(hv.value_new), torch.from_numpy(slots).cuda(),
                        _dev_u8(hv.k_scales), _dev_u8(hv.v_scales))
    torch.cuda.synchronize()
    kref, vref = hv.key_cache.copy(), hv.value_cache.copy()
    oracle.cache_write_fp8(kref, vref, kn, hv.value_new, slots, hv.k_scales, hv.v_scales)
    assert np.array_equal(kc.cpu().numpy(), kref)
    assert np.array_equal(vc.cpu().numpy(), vref)
    assert (kref == 0x7E).any() or (kref == 0xFE).any()   # saturation was exercised


def test_fp8_step_write_then_decode(pkv):
    import torch
    wl = W.custom_workload(4, 32, 8, 128, [1, 17, 64, 700], dtype="bf16", seed=3)
    hv = W.fp8_host_values(wl)
    kc, vc = _dev_u8(hv.key_cache), _dev_u8(hv.value_cache)
    ks, vs = _dev_u8(hv.k_scales), _dev_u8(hv.v_scales)
    pkv.cache_write_fp8(kc, vc, _bf16(hv.key_new), _bf16(hv.value_new),
                        torch.from_numpy(wl.slot_mapping).cuda(), ks, vs)
    out = pkv.decode_fp8(_bf16(hv.query), kc, vc, ks, vs, torch.from_numpy(wl.block_tables).cuda(),
                         torch.from_numpy(wl.step_context_lens).cuda(), wl.scale)
    torch.cuda.synchronize()
    kref, vref = hv.key_cache.copy(), hv.value_cache.copy()
    oracle.cache_write_fp8(kref, vref, hv.key_new, hv.value_new, wl.slot_mapping, hv.k_scales,
                           hv.v_scales)
    ref = oracle.paged_decode(hv.query, kref, vref, wl.block_tables, wl.step_context_lens,
                              wl.scale, k_scales=hv.k_scales, v_scales=hv.v_scales)
    H.assert_close(H.as_f64(out), ref, "bf16", "fp8 step")


def test_block_copy_fp8_bit_exact(pkv):
    import torch
    wl = W.custom_workload(3, 8, 8, 128, [40, 70, 5], dtype="bf16", seed=4, spare_blocks=6)
    hv = W.fp8_host_values(wl, poison_unused=False)
    used = set(wl.block_tables[wl.block_tables >= 0].tolist())
    free = [b for b in range(wl.num_blocks) if b not in used]
    pairs = np.array([[wl.block_tables[0, 2], free[0]], [wl.block_tables[1, 4], free[1]]],
                     dtype=np.int32)
    kc, vc = _dev_u8(hv.key_cache), _dev_u8(hv.value_cache)
    pkv.block_copy(kc, vc, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    kref, vref = hv.key_cache.copy(), hv.value_cache.copy()
    oracle.block_copy(kref, vref, pairs)
    assert np.array_equal(kc.cpu().numpy(), kref) and np.array_equal(vc.cpu().numpy(), vref)


@pytest.mark.parametrize("name", ["llama7b_mha", "llama70b_gqa", "long_splitk", "shared_prefix"])
def test_fp8_full_size_workload_sampled(pkv, name):
    import torch
    wl = W.make_workload(name)
    q, kc, vc, kn, vn, ks, vs = W.fp8_device_values(wl, "cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    lens = wl.context_lens
    out = pkv.decode_fp8(q, kc, vc, ks, vs, bt, torch.from_numpy(lens).cuda(), wl.scale,
                         partition_size=wl.partition_size)
    torch.cuda.synchronize()
    seqs, pairs = H.sample_pairs(wl, lens, n_seqs=5, heads_per_seq=4, seed=3)
    kch, vch, tabs, slens = H.compact_for_sequences(wl, seqs, kc, vc, lens)
    qh = H.device_to_host_bits(q[torch.as_tensor(seqs, device="cuda")])
    ref = oracle.paged_decode(qh, kch, vch, tabs, slens, wl.scale, sel=pairs, threads=8,
                              k_scales=ks.cpu().numpy(), v_scales=vs.cpu().numpy())
    got = np.stack([H.as_f64(out[seqs[i], h]) for i, h in pairs])
    H.assert_close(got, ref, "bf16", f"fp8 {name}")
