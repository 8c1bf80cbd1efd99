"""GPU parity: pa_decode_shared_prefix (prefix once per KV head, suffix per sequence,
merged) against the oracle on the full tables, and against pa_decode."""
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


def _shared_workload(B, hq, hkv, D, prefix_blocks, suffix_lens, seed):
    """Tables that all start with the same prefix_blocks blocks; context = prefix + suffix."""
    rng = np.random.default_rng(seed)
    lens = np.asarray([prefix_blocks * 16 + s for s in suffix_lens], np.int32)
    own = [-(-(int(L) + 1) // 16) - prefix_blocks for L in lens]
    own = [max(o, 0) for o in own]
    NB = prefix_blocks + sum(own) + 3
    perm = rng.permutation(NB).astype(np.int32)
    width = prefix_blocks + max(own + [0])
    tables = np.full((B, max(width, 1)), -1, np.int32)
    tables[:, :prefix_blocks] = perm[:prefix_blocks]
    pos = prefix_blocks
    for b in range(B):
        tables[b, prefix_blocks:prefix_blocks + own[b]] = perm[pos:pos + own[b]]
        pos += own[b]
    wl = W.Workload("shared_custom", B, hq, hkv, D, "bf16", 1.0, lens, tables, NB,
                    np.zeros(B, np.int64), seed=seed)
    return wl


def _run(pkv, wl, hv, n_prefix, lens=None, status=None, partition_size=0):
    import torch
    q = H.host_to_device(hv.query, torch.bfloat16)
    kc = H.host_to_device(hv.key_cache, torch.bfloat16)
    vc = H.host_to_device(hv.value_cache, torch.bfloat16)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(np.asarray(wl.context_lens if lens is None else lens, np.int32)).cuda()
    out = pkv.decode_shared_prefix(q, kc, vc, bt, cl, n_prefix, wl.scale, status=status,
                                   partition_size=partition_size)
    ref_gpu = pkv.decode(q, kc, vc, bt, cl, wl.scale)
    torch.cuda.synchronize()
    return out, ref_gpu


@pytest.mark.parametrize("hq,hkv,D", [(8, 8, 128), (32, 8, 128), (16, 2, 128), (12, 4, 64),
                                      (32, 2, 128), (4, 4, 64), (16, 8, 128)])
@pytest.mark.parametrize("prefix_blocks", [1, 7, 40])
def test_shared_prefix_matches_oracle(pkv, hq, hkv, D, prefix_blocks):
    suffix = [0, 1, 15, 16, 17, 200, 640, 3]
    wl = _shared_workload(len(suffix), hq, hkv, D, prefix_blocks, suffix, seed=hq + D + prefix_blocks)
    hv = W.host_values(wl)              # slots holding no context token are NaN
    out, ref_gpu = _run(pkv, wl, hv, prefix_blocks)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                              wl.context_lens, wl.scale, threads=4)
    H.assert_close(H.as_f64(out), ref, "bf16", f"shared prefix {hq}/{hkv}/{D} n={prefix_blocks}")
    H.assert_close(H.as_f64(out), H.as_f64(ref_gpu), "bf16", "shared prefix vs pa_decode")


def test_many_sequences_span_several_row_tiles(pkv):
    """70 sequences x 4 heads of a group = 280 rows per KV head: two 256-row
    tiles on the tensor-core prefix path, the second one partly empty."""
    rng = np.random.default_rng(12)
    suffix = rng.integers(0, 300, 70).tolist()
    wl = _shared_workload(70, 8, 2, 128, 19, suffix, seed=13)
    hv = W.host_values(wl)
    out, ref_gpu = _run(pkv, wl, hv, 19)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                              wl.context_lens, wl.scale, threads=8)
    H.assert_close(H.as_f64(out), ref, "bf16", "70 sequences")


@pytest.mark.parametrize("hq,hkv,partition_size", [(16, 2, 0), (16, 4, 0), (8, 4, 32), (16, 8, 16)])
def test_many_short_suffixes(pkv, hq, hkv, partition_size):
    """Hundreds of short suffixes (some empty) and, with small partitions,
    several partitions per sequence: more suffix CTAs than fit on the GPU at
    once, and empty trailing partitions."""
    rng = np.random.default_rng(hq * 100 + hkv + partition_size)
    B = 600
    suffix = rng.integers(0, 90, B)
    suffix[::7] = 0
    wl = _shared_workload(B, hq, hkv, 128, 3, suffix.tolist(), seed=hq + hkv + partition_size)
    hv = W.host_values(wl)
    out, ref_gpu = _run(pkv, wl, hv, 3, partition_size=partition_size)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                              wl.context_lens, wl.scale, threads=8)
    H.assert_close(H.as_f64(out), ref, "bf16", f"{B} suffixes {hq}/{hkv} P={partition_size}")
    H.assert_close(H.as_f64(out), H.as_f64(ref_gpu), "bf16", "many suffixes vs pa_decode")


def test_contexts_shorter_than_the_prefix_are_masked(pkv):
    wl = _shared_workload(4, 16, 4, 128, 10, [5, 0, 30, 1], seed=9)
    hv = W.host_values(wl, poison_unused=False)
    lens = wl.context_lens.copy()
    lens[1] = 37            # ends inside the prefix
    lens[3] = 0             # empty
    out, _ = _run(pkv, wl, hv, 10, lens=lens, partition_size=64)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables, lens,
                              wl.scale)
    got = H.as_f64(out)
    assert np.all(got[3] == 0)
    H.assert_close(got, ref, "bf16", "short contexts")


def test_prefix_mismatch_is_flagged(pkv):
    import torch
    wl = _shared_workload(4, 8, 8, 128, 6, [10, 20, 30, 40], seed=4)
    hv = W.host_values(wl, poison_unused=False)
    wl.block_tables[2, 3] = wl.block_tables[2, 6]    # row 2 leaves the shared prefix
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _run(pkv, wl, hv, 6, status=status)
    assert int(status.item()) & pkv._lib.PA_DEV_PREFIX_MISMATCH


@pytest.mark.parametrize("cow", [False, True])
def test_shared_prefix_workload_full_size(pkv, cow):
    """The 128-sequence mix: before copy-on-write all 64 prefix blocks are shared;
    after it the first 16 sequences own block 63, so 63 blocks are shared."""
    import torch
    wl = W.make_workload("shared_prefix")
    if not cow:
        wl.block_tables[:wl.cow_pairs.shape[0], 63] = wl.cow_pairs[0, 0]
    n_prefix = pkv.shared_prefix_blocks(wl.block_tables)
    assert n_prefix == (63 if cow else 64)
    q, kc, vc, kn, vn = W.device_values(wl, "cuda")
    if cow:
        pkv.block_copy(kc, vc, torch.from_numpy(wl.cow_pairs).cuda())
    bt = torch.from_numpy(wl.block_tables).cuda()
    lens = wl.step_context_lens
    cl = torch.from_numpy(lens).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.decode_shared_prefix(q, kc, vc, bt, cl, n_prefix, wl.scale, status=status)
    plain = pkv.decode(q, kc, vc, bt, cl, wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    H.assert_close(H.as_f64(out), H.as_f64(plain), "bf16", "cascade vs plain decode")
    seqs, pairs = H.sample_pairs(wl, lens, n_seqs=5, heads_per_seq=4, seed=4)
    kch, vch, tabs, slens = H.compact_for_sequences(wl, seqs, kc, vc, lens)
    qh = H.device_to_host_bits(q[torch.as_tensor(seqs, device="cuda")])
    ref = oracle.paged_decode(qh, kch, vch, tabs, slens, wl.scale, sel=pairs, threads=8)
    got = np.stack([H.as_f64(out[seqs[i], h]) for i, h in pairs])
    H.assert_close(got, ref, "bf16", "shared-prefix workload")


@pytest.mark.parametrize("fill", ["zeros", "ones", "random"])
def test_workspace_reused_across_calls(pkv, fill):
    """The CTA that completes a row set merges it, counted on per-(sequence, KV
    head) words in the workspace.  Whatever the workspace held before (zeros,
    all-ones bytes, random bytes) and however often it is reused, every call
    must give the same result as pa_decode."""
    import torch
    rng = np.random.default_rng(31)
    suffix = rng.integers(0, 400, 40).tolist()
    wl = _shared_workload(40, 16, 4, 128, 21, suffix, seed=32)
    hv = W.host_values(wl, poison_unused=False)
    q = H.host_to_device(hv.query, torch.bfloat16)
    kc = H.host_to_device(hv.key_cache, torch.bfloat16)
    vc = H.host_to_device(hv.value_cache, torch.bfloat16)
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(wl.context_lens).cuda()
    need = pkv.lib().pa_decode_shared_prefix_workspace_bytes(40, 16, 4, 128, wl.block_tables.shape[1],
                                                             21, 64)
    if fill == "zeros":
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    elif fill == "ones":
        ws = torch.full((need,), 255, dtype=torch.uint8, device="cuda")
    else:
        g = torch.Generator(device="cuda")
        g.manual_seed(5)
        ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda", generator=g)
    plain = pkv.decode(q, kc, vc, bt, cl, wl.scale)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(3):
        out = pkv.decode_shared_prefix(q, kc, vc, bt, cl, 21, wl.scale, workspace=ws, status=status,
                                       partition_size=64)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        H.assert_close(H.as_f64(out), H.as_f64(plain), "bf16", f"call {call} ({fill})")


def _fp8_run(pkv, wl, hv, n_prefix, lens=None, status=None, partition_size=0, workspace=None):
    import torch
    q = H.host_to_device(hv.query, torch.bfloat16)
    kc = torch.from_numpy(np.ascontiguousarray(hv.key_cache)).cuda()
    vc = torch.from_numpy(np.ascontiguousarray(hv.value_cache)).cuda()
    ks = torch.from_numpy(np.ascontiguousarray(hv.k_scales)).cuda()
    vs = torch.from_numpy(np.ascontiguousarray(hv.v_scales)).cuda()
    bt = torch.from_numpy(wl.block_tables).cuda()
    cl = torch.from_numpy(np.asarray(wl.context_lens if lens is None else lens, np.int32)).cuda()
    out = pkv.decode_shared_prefix_fp8(q, kc, vc, ks, vs, bt, cl, n_prefix, wl.scale, status=status,
                                       partition_size=partition_size, workspace=workspace)
    ref_gpu = pkv.decode_fp8(q, kc, vc, ks, vs, bt, cl, wl.scale)
    torch.cuda.synchronize()
    return out, ref_gpu


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 8), (16, 2), (16, 8), (6, 2)])
@pytest.mark.parametrize("prefix_blocks", [1, 9, 40])
def test_shared_prefix_fp8_matches_oracle(pkv, hq, hkv, prefix_blocks):
    """E4M3 pools: the prefix widened to bf16 code values on the tensor cores with
    the per-head scales folded in, the suffix on the FP8 decode kernel (group 3
    takes plain FP8 decode)."""
    suffix = [0, 1, 15, 16, 17, 200, 640, 3]
    wl = _shared_workload(len(suffix), hq, hkv, 128, prefix_blocks, suffix, seed=hq + hkv + prefix_blocks)
    hv = W.fp8_host_values(wl)          # slots holding no context token carry the NaN code
    out, ref_gpu = _fp8_run(pkv, wl, hv, prefix_blocks)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                              wl.context_lens, wl.scale, threads=4, k_scales=hv.k_scales,
                              v_scales=hv.v_scales)
    H.assert_close(H.as_f64(out), ref, "bf16", f"fp8 shared prefix {hq}/{hkv} n={prefix_blocks}")
    H.assert_close(H.as_f64(out), H.as_f64(ref_gpu), "bf16", "fp8 shared prefix vs pa_decode_fp8")


@pytest.mark.parametrize("hq,hkv,partition_size", [(16, 4, 0), (16, 2, 32)])
def test_shared_prefix_fp8_many_short_suffixes(pkv, hq, hkv, partition_size):
    """E4M3 pools with hundreds of short suffixes (more CTAs than fit at once)."""
    rng = np.random.default_rng(7 * hq + hkv + partition_size)
    B = 500
    suffix = rng.integers(0, 90, B)
    suffix[::5] = 0
    wl = _shared_workload(B, hq, hkv, 128, 2, suffix.tolist(), seed=3 * hq + hkv)
    hv = W.fp8_host_values(wl)
    out, ref_gpu = _fp8_run(pkv, wl, hv, 2, partition_size=partition_size)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                              wl.context_lens, wl.scale, threads=8, k_scales=hv.k_scales,
                              v_scales=hv.v_scales)
    H.assert_close(H.as_f64(out), ref, "bf16", f"fp8 {B} suffixes {hq}/{hkv} P={partition_size}")
    H.assert_close(H.as_f64(out), H.as_f64(ref_gpu), "bf16", "fp8 many suffixes vs pa_decode_fp8")


def test_shared_prefix_fp8_short_contexts_and_split_suffix(pkv):
    wl = _shared_workload(6, 16, 4, 128, 12, [5, 0, 30, 1, 900, 333], seed=19)
    hv = W.fp8_host_values(wl, poison_unused=False)
    lens = wl.context_lens.copy()
    lens[1] = 37            # ends inside the prefix
    lens[3] = 0             # empty
    out, _ = _fp8_run(pkv, wl, hv, 12, lens=lens, partition_size=64)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables, lens,
                              wl.scale, k_scales=hv.k_scales, v_scales=hv.v_scales)
    got = H.as_f64(out)
    assert np.all(got[3] == 0)
    H.assert_close(got, ref, "bf16", "fp8 short contexts")


def test_shared_prefix_fp8_workload_full_size(pkv):
    """The 128-sequence mix on E4M3 pools, after copy-on-write (63 shared blocks)."""
    import torch
    wl = W.make_workload("shared_prefix")
    n_prefix = pkv.shared_prefix_blocks(wl.block_tables)
    q, kc, vc, _, _, ks, vs = W.fp8_device_values(wl, "cuda")
    pkv.block_copy(kc, vc, torch.from_numpy(wl.cow_pairs).cuda())
    bt = torch.from_numpy(wl.block_tables).cuda()
    lens = wl.step_context_lens
    cl = torch.from_numpy(lens).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.decode_shared_prefix_fp8(q, kc, vc, ks, vs, bt, cl, n_prefix, wl.scale, status=status)
    plain = pkv.decode_fp8(q, kc, vc, ks, vs, bt, cl, wl.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    H.assert_close(H.as_f64(out), H.as_f64(plain), "bf16", "fp8 cascade vs plain FP8 decode")


@pytest.mark.parametrize("lo,hi", [(288, 320), (320, 384), (600, 700)])
def test_prefix_scores_rising_in_later_tiles(pkv, lo, hi):
    """Keys of the shared prefix scaled up at [lo, hi): the prefix kernel's rows see
    their scores jump in a later K/V tile and move their reference there."""
    suffix = [0, 1, 15, 200, 640, 3, 90, 33]
    wl = _shared_workload(len(suffix), 32, 8, 128, 48, suffix, seed=lo)
    hv = W.host_values(wl)
    k = W.bf16_bits_to_f32(hv.key_cache)
    for pos in range(lo, hi):
        phys = int(wl.block_tables[0, pos // 16])
        k[phys, :, pos % 16] *= np.float32(8.0)
    hv.key_cache = np.where(np.isnan(k), hv.key_cache, W.to_bf16_bits(k))
    out, ref_gpu = _run(pkv, wl, hv, 48)
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                              wl.context_lens, wl.scale, threads=4)
    H.assert_close(H.as_f64(out), ref, "bf16", f"prefix keys x8 at [{lo}, {hi})")
    H.assert_close(H.as_f64(out), H.as_f64(ref_gpu), "bf16", "against pa_decode")
