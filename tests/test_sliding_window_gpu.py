"""GPU parity for sliding-window decode: pa_decode_sliding_window through the C ABI
against the fp64 oracle with the same window.

Every slot before each sequence's window is poisoned (NaN, or the E4M3 NaN code)
and every table entry wholly before it is set to -1, as a block manager that
released those blocks leaves it: a kernel that reads outside the window shows
it as NaN in the output or as a device status bit."""
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


def _window_start(L, window):
    return L - window if L > window else 0


def _poison_before_window(wl, hv, window, nan_code):
    """Poison the slots of positions [0, L - window) and drop the dead blocks
    from the tables (entry -1); returns the trimmed tables."""
    tables = wl.block_tables.copy()
    for b in range(wl.num_seqs):
        L = int(wl.context_lens[b])
        start = _window_start(L, window)
        for t in range(start):
            phys = int(tables[b, t // 16])
            hv.key_cache[phys, :, t % 16, :] = nan_code
            hv.value_cache[phys, :, t % 16, :] = nan_code
        for j in range(start // 16):
            tables[b, j] = -1
    return tables


def _nan_of(wl):
    return np.uint16(0x7FC0) if wl.dtype == "bf16" else np.float32(np.nan)


def _run(pkv, wl, hv, tables, window, partition_size=0, fp8=False):
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.from_numpy(tables).cuda()
    cl = torch.from_numpy(np.asarray(wl.context_lens, np.int32)).cuda()
    if fp8:
        u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        out = pkv.decode_sliding_window(
            H.host_to_device(hv.query, torch.bfloat16), u8(hv.key_cache), u8(hv.value_cache),
            bt, cl, window, wl.scale, k_scales=u8(hv.k_scales), v_scales=u8(hv.v_scales),
            partition_size=partition_size, status=status)
    else:
        dt = H.torch_dtype(wl)
        out = pkv.decode_sliding_window(
            H.host_to_device(hv.query, dt), H.host_to_device(hv.key_cache, dt),
            H.host_to_device(hv.value_cache, dt), bt, cl, window, wl.scale,
            partition_size=partition_size, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


def _oracle(wl, hv, tables, window, fp8=False):
    extra = dict(k_scales=hv.k_scales, v_scales=hv.v_scales) if fp8 else {}
    return oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, tables,
                               np.asarray(wl.context_lens, np.int32), wl.scale, threads=4,
                               window=window, **extra)


LENS = [0, 1, 15, 16, 17, 40, 100, 513, 1100]


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (8, 8, 64), (8, 2, 128), (32, 2, 128),
                                      (12, 4, 64)])
@pytest.mark.parametrize("window", [1, 16, 17, 40, 257, 4096])
@pytest.mark.parametrize("partition_size", [0, 32])
def test_bf16_window_matches_oracle(pkv, hq, hkv, d, window, partition_size):
    wl = W.custom_workload(len(LENS), hq, hkv, d, LENS, dtype="bf16", seed=hq + d + window)
    hv = W.host_values(wl)
    tables = _poison_before_window(wl, hv, window, _nan_of(wl))
    got = H.as_f64(_run(pkv, wl, hv, tables, window, partition_size))
    H.assert_close(got, _oracle(wl, hv, tables, window), "bf16",
                   f"bf16 {hq}/{hkv}/{d} W={window} P={partition_size}")


@pytest.mark.parametrize("d", [32, 128, 256])
@pytest.mark.parametrize("window", [1, 33, 300])
def test_fp32_window_matches_oracle(pkv, d, window):
    wl = W.custom_workload(len(LENS), 4, 2, d, LENS, dtype="f32", seed=d + window)
    hv = W.host_values(wl)
    tables = _poison_before_window(wl, hv, window, _nan_of(wl))
    for ps in (0, 16):
        got = H.as_f64(_run(pkv, wl, hv, tables, window, ps))
        H.assert_close(got, _oracle(wl, hv, tables, window), "f32", f"f32 d={d} W={window} P={ps}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2), (12, 4)])
@pytest.mark.parametrize("window", [1, 24, 300])
def test_fp8_window_matches_oracle(pkv, hq, hkv, window):
    wl = W.custom_workload(len(LENS), hq, hkv, 128, LENS, dtype="bf16", seed=hq * hkv + window)
    hv = W.fp8_host_values(wl)
    tables = _poison_before_window(wl, hv, window, np.uint8(0x7F))
    for ps in (0, 48):
        got = H.as_f64(_run(pkv, wl, hv, tables, window, ps, fp8=True))
        H.assert_close(got, _oracle(wl, hv, tables, window, fp8=True), "bf16",
                       f"fp8 {hq}/{hkv} W={window} P={ps}")


def test_window_at_least_the_context_equals_plain_decode(pkv):
    import torch
    wl = W.custom_workload(len(LENS), 8, 2, 128, LENS, dtype="bf16", seed=11)
    hv = W.host_values(wl)
    plain = pkv.decode(H.host_to_device(hv.query, torch.bfloat16),
                       H.host_to_device(hv.key_cache, torch.bfloat16),
                       H.host_to_device(hv.value_cache, torch.bfloat16),
                       torch.from_numpy(wl.block_tables).cuda(),
                       torch.from_numpy(np.asarray(wl.context_lens, np.int32)).cuda(), wl.scale,
                       partition_size=64)
    windowed = _run(pkv, wl, hv, wl.block_tables, max(LENS), partition_size=64)
    # same partitions, same order of accumulation: identical bits
    assert torch.equal(plain.view(torch.int16), windowed.view(torch.int16))


def test_window_one_is_exactly_the_last_v_row(pkv):
    """softmax over one score is 1: the output is that row of V, rounded to bf16."""
    wl = W.custom_workload(len(LENS), 8, 2, 128, LENS, dtype="bf16", seed=12)
    hv = W.host_values(wl)
    tables = _poison_before_window(wl, hv, 1, _nan_of(wl))
    got = H.device_to_host_bits(_run(pkv, wl, hv, tables, 1))
    for b, L in enumerate(LENS):
        for h in range(8):
            if L == 0:
                assert not np.any(got[b, h] & 0x7FFF)
                continue
            phys = int(wl.block_tables[b, (L - 1) // 16])
            assert np.array_equal(got[b, h], hv.value_cache[phys, h // 4, (L - 1) % 16])


def test_trimmed_block_manager_tables_decode_through_the_window(pkv):
    """The block manager's trim_window releases what the windowed decode never reads."""
    import torch
    window, NB, HKV, HQ, D = 50, 64, 2, 8, 128
    bm = pkv.BlockManager(NB)
    lens = [130, 47, 300]
    for s, n in enumerate(lens):
        bm.alloc_seq(s, n)
    released = sum(bm.trim_window(s, window) for s in range(3))
    assert released == sum(max(n - window, 0) // 16 for n in lens)
    tables, cl = bm.fill_tables(list(range(3)), 20)
    assert (tables[:, 0] == -1).sum() == 2
    rng = np.random.default_rng(1)
    kc = W.to_bf16_bits(rng.standard_normal((NB, HKV, 16, D), dtype=np.float32))
    vc = W.to_bf16_bits(rng.standard_normal((NB, HKV, 16, D), dtype=np.float32))
    q = W.to_bf16_bits(rng.standard_normal((3, HQ, D), dtype=np.float32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.decode_sliding_window(
        H.host_to_device(q, torch.bfloat16), H.host_to_device(kc, torch.bfloat16),
        H.host_to_device(vc, torch.bfloat16), torch.from_numpy(tables).cuda(),
        torch.from_numpy(cl).cuda(), window, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.paged_decode(q, kc, vc, tables, cl, 1 / np.sqrt(D), window=window)
    H.assert_close(H.as_f64(out), ref, "bf16", "trimmed tables")
