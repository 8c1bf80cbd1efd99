"""GPU parity: pa_decode through the C ABI against the fp64 oracle."""
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


def _device_inputs(wl, hv, lens=None):
    import torch
    dt = H.torch_dtype(wl)
    q = H.host_to_device(hv.query, dt)
    kc = H.host_to_device(hv.key_cache, dt)
    vc = H.host_to_device(hv.value_cache, dt)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(np.asarray(wl.context_lens if lens is None else lens, np.int32)).cuda()
    return q, kc, vc, bt, cl


def _run(pkv, wl, hv, lens=None, partition_size=0, status=None, scale=None):
    import torch
    q, kc, vc, bt, cl = _device_inputs(wl, hv, lens)
    out = pkv.decode(q, kc, vc, bt, cl, wl.scale if scale is None else scale,
                     partition_size=partition_size, status=status)
    torch.cuda.synchronize()
    return out


def _oracle(wl, hv, lens=None, scale=None):
    lens = wl.context_lens if lens is None else lens
    return oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                               np.asarray(lens, np.int32), wl.scale if scale is None else scale,
                               threads=4)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (16, 2)])
@pytest.mark.parametrize("scale", [-0.0883883, 0.0])
def test_nonpositive_scale(pkv, hq, hkv, scale):
    """A negative scale reverses the order of the scores; scale 0 weighs every
    position equally (MHA and GQA consumers, split and unsplit)."""
    lens = [1, 17, 300, 1100]
    wl = W.custom_workload(len(lens), hq, hkv, 128, lens, dtype="bf16", seed=hq + hkv)
    hv = W.host_values(wl)
    for ps in (0, 64):
        got = H.as_f64(_run(pkv, wl, hv, partition_size=ps, scale=scale))
        H.assert_close(got, _oracle(wl, hv, scale=scale), "bf16", f"decode scale {scale} P {ps}")


def test_tiny_fp32_workload(pkv):
    wl = W.make_workload("tiny")
    hv = W.host_values(wl)                       # unused slots hold NaN
    got = H.as_f64(_run(pkv, wl, hv))
    H.assert_close(got, _oracle(wl, hv), "f32", "tiny decode")


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 128), (8, 8, 64), (8, 2, 128), (16, 2, 128),
                                      (8, 1, 64), (12, 4, 128), (32, 2, 128), (6, 3, 64),
                                      (4, 4, 64)])
@pytest.mark.parametrize("partition_size", [0, 64, 16384])
def test_random_bf16_shapes(pkv, hq, hkv, d, partition_size):
    lens = [1, 15, 16, 17, 100, 513, 1100]
    wl = W.custom_workload(len(lens), hq, hkv, d, lens, dtype="bf16", seed=hq * 7 + d)
    hv = W.host_values(wl)
    got = H.as_f64(_run(pkv, wl, hv, partition_size=partition_size))
    H.assert_close(got, _oracle(wl, hv), "bf16", f"bf16 {hq}/{hkv}/{d} P={partition_size}")


@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_random_fp32_shapes(pkv, d):
    lens = [1, 16, 33, 200, 700]
    wl = W.custom_workload(len(lens), 4, 2, d, lens, dtype="f32", seed=d)
    hv = W.host_values(wl)
    for ps in (0, 32):
        got = H.as_f64(_run(pkv, wl, hv, partition_size=ps))
        H.assert_close(got, _oracle(wl, hv), "f32", f"f32 d={d} P={ps}")


@pytest.mark.parametrize("hq,hkv", [(4, 4), (16, 2)])
def test_one_token_context_is_exactly_v(pkv, hq, hkv):
    wl = W.custom_workload(5, hq, hkv, 128, [1] * 5, dtype="bf16", seed=3)
    hv = W.host_values(wl)
    got = H.device_to_host_bits(_run(pkv, wl, hv))
    g = hq // hkv
    for b in range(5):
        phys = wl.block_tables[b, 0]
        for h in range(hq):
            assert np.array_equal(got[b, h], hv.value_cache[phys, h // g, 0])


def test_empty_context_gives_zeros(pkv):
    wl = W.custom_workload(3, 8, 2, 128, [0, 5, 0], dtype="bf16", seed=4)
    hv = W.host_values(wl)
    got = H.as_f64(_run(pkv, wl, hv))
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    H.assert_close(got, _oracle(wl, hv), "bf16", "empty contexts")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 4)])
def test_permuting_physical_blocks_is_bit_identical(pkv, hq, hkv):
    lens = [3, 40, 257, 600]
    wl = W.custom_workload(4, hq, hkv, 128, lens, dtype="bf16", seed=5, spare_blocks=9)
    hv = W.host_values(wl)
    ref = H.device_to_host_bits(_run(pkv, wl, hv, partition_size=128))
    perm = np.random.default_rng(1).permutation(wl.num_blocks)
    kc2 = np.empty_like(hv.key_cache)
    vc2 = np.empty_like(hv.value_cache)
    kc2[perm] = hv.key_cache
    vc2[perm] = hv.value_cache
    wl.block_tables = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)],
                               -1).astype(np.int32)
    hv2 = W.HostValues(hv.query, kc2, vc2, hv.key_new, hv.value_new)
    got = H.device_to_host_bits(_run(pkv, wl, hv2, partition_size=128))
    assert np.array_equal(got, ref)


def test_gqa_path_equals_mha_path_on_repeated_heads(pkv):
    lens = [30, 300, 1000]
    wl = W.custom_workload(3, 16, 2, 128, lens, dtype="bf16", seed=6)
    hv = W.host_values(wl)
    gqa = H.as_f64(_run(pkv, wl, hv))
    wl_mha = W.custom_workload(3, 16, 2, 128, lens, dtype="bf16", seed=6)
    wl_mha.num_kv_heads = 16
    hv_mha = W.HostValues(hv.query, np.repeat(hv.key_cache, 8, axis=1),
                          np.repeat(hv.value_cache, 8, axis=1), hv.key_new, hv.value_new)
    mha = H.as_f64(_run(pkv, wl_mha, hv_mha))
    H.assert_close(gqa, mha, "bf16", "GQA vs MHA")
    H.assert_close(gqa, _oracle(wl, hv), "bf16", "GQA vs oracle")


def test_out_of_range_indices_are_flagged_not_followed(pkv):
    import torch
    lens = [20, 40]
    wl = W.custom_workload(2, 4, 4, 128, lens, dtype="bf16", seed=7)
    hv = W.host_values(wl, poison_unused=False)
    wl.block_tables[1, 1] = wl.num_blocks + 1000          # out of the pool
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _run(pkv, wl, hv, status=status)
    assert int(status.item()) & pkv._lib.PA_DEV_BAD_BLOCK_ID
    status.zero_()
    bad_lens = np.array([20, wl.max_blocks * 16 + 50], np.int32)
    out = _run(pkv, wl, hv, lens=bad_lens, status=status)
    assert int(status.item()) & pkv._lib.PA_DEV_BAD_CONTEXT_LEN
    assert torch.isfinite(out[0].float()).all()


def test_launch_counter_counts_decode_kernels(pkv):
    lens = [2000, 30]
    wl = W.custom_workload(2, 4, 4, 128, lens, dtype="bf16", seed=8)
    hv = W.host_values(wl)
    n0 = pkv.launch_count()
    _run(pkv, wl, hv, partition_size=512)          # split: decode + reduce
    assert pkv.launch_count() - n0 == 2
    n1 = pkv.launch_count()
    _run(pkv, wl, hv, partition_size=16384)        # one partition: decode only
    assert pkv.launch_count() - n1 == 1


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the bench uses, checked on
# sampled (sequence, head) pairs the oracle computes one by one.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["llama7b_mha", "llama70b_gqa", "long_splitk", "shared_prefix"])
def test_full_size_workload_sampled(pkv, name):
    import torch
    wl = W.make_workload(name)
    q, kc, vc, kn, vn = W.device_values(wl, "cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    lens = wl.context_lens
    cl = torch.from_numpy(lens).cuda()
    out = pkv.decode(q, kc, vc, bt, cl, wl.scale, partition_size=wl.partition_size)
    torch.cuda.synchronize()
    seqs, pairs = H.sample_pairs(wl, lens, n_seqs=6, heads_per_seq=4, seed=1)
    kch, vch, tabs, slens = H.compact_for_sequences(wl, seqs, kc, vc, lens)
    qh = H.device_to_host_bits(q[torch.as_tensor(seqs, device="cuda")])
    ref = oracle.paged_decode(qh, kch, vch, tabs, slens, wl.scale, sel=pairs, threads=8)
    got = np.stack([H.as_f64(out[seqs[i], h]) for i, h in pairs])
    H.assert_close(got, ref, "bf16", name)
    assert torch.isfinite(out.float()).all()
