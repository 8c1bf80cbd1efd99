"""Pins for the oracle: each test ties it to something other than itself.

* an independent library routine on the same tokens laid out contiguously
  (torch's scaled_dot_product_attention in fp64);
* closed forms (one-token context, constant values, zero query, a dominant key);
* invariances the pages state (paging does not change the arithmetic, so
  permuting physical block ids changes nothing; GQA equals MHA with the KV heads
  repeated);
* the worked block-table examples printed on the pages (tests/golden).

None of these tests touches a GPU or the CUDA library.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _scatter(contig_k, contig_v, tables, lens, num_blocks, fill=np.nan):
    """Place each sequence's contiguous K/V rows [Hkv][L][D] into a paged pool."""
    Hkv, D = contig_k[0].shape[0], contig_k[0].shape[2]
    kc = np.full((num_blocks, Hkv, 16, D), fill, dtype=np.float32)
    vc = np.full((num_blocks, Hkv, 16, D), fill, dtype=np.float32)
    for b, L in enumerate(lens):
        for t in range(L):
            phys = tables[b][t // 16]
            kc[phys, :, t % 16, :] = contig_k[b][:, t, :]
            vc[phys, :, t % 16, :] = contig_v[b][:, t, :]
    return kc, vc


def _random_paged(rng, B, Hq, Hkv, D, lens, spare=3):
    need = [-(-L // 16) for L in lens]
    NB = sum(need) + spare
    perm = rng.permutation(NB)
    tables = np.full((B, max(max(need), 1)), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        tables[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    ck = [rng.standard_normal((Hkv, L, D)).astype(np.float32) for L in lens]
    cv = [rng.standard_normal((Hkv, L, D)).astype(np.float32) for L in lens]
    kc, vc = _scatter(ck, cv, tables, lens, NB)
    return q, ck, cv, kc, vc, tables, np.asarray(lens, dtype=np.int32)


def _sdpa(q, ck, cv, scale, group):
    """Library attention over contiguous tokens: q [Hq][D], k/v [Hkv][L][D] -> [Hq][D]."""
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]       # [1,Hq,1,D]
    kt = torch.from_numpy(ck.astype(np.float64))[None]                  # [1,Hkv,L,D]
    vt = torch.from_numpy(cv.astype(np.float64))[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale,
                                                         enable_gqa=group > 1)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,scale", [
    (4, 4, 4, 64, [1, 17, 33, 64], 0.125),
    (3, 8, 2, 128, [15, 16, 100], 0.0883883),
    (2, 16, 2, 64, [31, 48], 0.3),
    (2, 6, 3, 32, [5, 250], 1.7),
])
def test_matches_library_attention_on_contiguous_tokens(B, Hq, Hkv, D, lens, scale):
    rng = np.random.default_rng(1234 + B * Hq + D)
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, B, Hq, Hkv, D, lens)
    got = oracle.paged_decode(q, kc, vc, tables, L, scale)
    for b in range(B):
        want = _sdpa(q[b], ck[b], cv[b], scale, Hq // Hkv)
        np.testing.assert_allclose(got[b], want, rtol=1e-11, atol=1e-12)


def test_tiny_workload_matches_brute_force_loops():
    """The tiny fp32 workload (4 sequences of 1, 17, 33 and 64 tokens, 4 heads,
    head_dim 64, a 16-block pool in shuffled order) against attention written
    out as plain Python loops: each token found through its sequence's table
    entry t // 16 at slot t % 16, scores, the largest one, exponentials, their
    sum, the weighted values."""
    import math
    wl = W.make_workload("tiny")
    hv = W.host_values(wl)
    lens = [int(x) for x in wl.context_lens]
    ref = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables,
                              wl.context_lens, wl.scale)
    D = wl.head_dim
    g = wl.num_q_heads // wl.num_kv_heads
    for b in range(wl.num_seqs):
        for h in range(wl.num_q_heads):
            kvh = h // g
            q = [float(x) for x in hv.query[b, h]]
            scores = []
            for t in range(lens[b]):
                phys = int(wl.block_tables[b, t // 16])
                k = hv.key_cache[phys, kvh, t % 16]
                s = 0.0
                for d in range(D):
                    s += q[d] * float(k[d])
                scores.append(s * wl.scale)
            top = max(scores)
            weights = [math.exp(s - top) for s in scores]
            total = sum(weights)
            for d in range(D):
                acc = 0.0
                for t in range(lens[b]):
                    phys = int(wl.block_tables[b, t // 16])
                    acc += weights[t] * float(hv.value_cache[phys, kvh, t % 16, d])
                assert abs(acc / total - ref[b, h, d]) <= 1e-12 * (1.0 + abs(acc / total)), (b, h, d)


def test_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, lens, scale = 2, 4, 2, 64, [9, 40], 0.125
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, B, Hq, Hkv, D, lens)
    qb, kcb, vcb = (W.to_bf16_bits(a) for a in (q, kc, vc))
    got = oracle.paged_decode(qb, kcb, vcb, tables, L, scale)

    def as_f64(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()

    for b in range(B):
        ckb = [as_f64(W.to_bf16_bits(x)) for x in ck]
        cvb = [as_f64(W.to_bf16_bits(x)) for x in cv]
        want = _sdpa(as_f64(qb[b]), ckb[b], cvb[b], scale, Hq // Hkv)
        np.testing.assert_allclose(got[b], want, rtol=1e-11, atol=1e-12)


def test_one_token_context_returns_its_value_exactly():
    rng = np.random.default_rng(3)
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 3, 4, 2, 64, [1, 1, 1])
    got = oracle.paged_decode(q, kc, vc, tables, L, 0.125)
    for b in range(3):
        for h in range(4):
            assert np.array_equal(got[b, h], cv[b][h // 2, 0, :].astype(np.float64))


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(4)
    lens = [7, 33, 130]
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 3, 4, 4, 64, lens)
    c = rng.standard_normal(64).astype(np.float32)
    cv = [np.broadcast_to(c, x.shape).copy() for x in cv]
    kc, vc = _scatter(ck, cv, tables, lens, kc.shape[0])
    got = oracle.paged_decode(q, kc, vc, tables, L, 0.125)
    np.testing.assert_allclose(got, np.broadcast_to(c.astype(np.float64), got.shape), rtol=1e-13,
                               atol=1e-13)


def test_zero_query_averages_the_context():
    rng = np.random.default_rng(5)
    lens = [1, 16, 17, 77]
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 4, 2, 2, 32, lens)
    got = oracle.paged_decode(np.zeros_like(q), kc, vc, tables, L, 0.5)
    for b, n in enumerate(lens):
        want = cv[b].astype(np.float64).mean(axis=1)        # [Hkv][D]
        np.testing.assert_allclose(got[b], want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("t_star", [0, 15, 16, 17, 63, 64, 99])
def test_dominant_key_selects_its_token(t_star):
    """A key aligned with q and far larger than the rest puts all weight on its token."""
    rng = np.random.default_rng(6)
    lens = [100]
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 1, 1, 1, 64, lens)
    ck[0] *= 0.01
    ck[0][0, t_star] = 40.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    kc, vc = _scatter(ck, cv, tables, lens, kc.shape[0])
    got = oracle.paged_decode(q, kc, vc, tables, L, 1.0)
    np.testing.assert_allclose(got[0, 0], cv[0][0, t_star], rtol=1e-9, atol=1e-9)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_worked_block_table_reads_only_its_session(golden_dir):
    """Session X of the pool diagram: tokens live in blocks 7, 2, 11, 5, 9 of a 12-block pool."""
    g = _load(golden_dir, "block_tables.json")["session_x"]
    table, owners, NB = g["table"], g["pool_owner"], g["pool_size"]
    L = 16 * len(table)
    kc = np.zeros((NB, 1, 16, 4), dtype=np.float32)
    vc = np.full((NB, 1, 16, 4), 1.0e6, dtype=np.float32)   # other sessions' and free blocks
    for t in range(L):
        phys = table[t // 16]
        assert owners[phys] == "X"
        vc[phys, 0, t % 16, :] = t                          # V of token t encodes t
    q = np.zeros((1, 1, 4), dtype=np.float32)
    got = oracle.paged_decode(q, kc, vc, np.array([table], np.int32), np.array([L], np.int32), 1.0)
    np.testing.assert_allclose(got[0, 0], np.full(4, (L - 1) / 2.0), rtol=0, atol=1e-12)
    # a dominant key on token 37 (position 2 -> block 11, offset 5) selects exactly it
    kc[11, 0, 5, :] = 50.0
    q1 = np.ones((1, 1, 4), dtype=np.float32)
    got = oracle.paged_decode(q1, kc, vc, np.array([table], np.int32), np.array([L], np.int32), 1.0)
    np.testing.assert_allclose(got[0, 0], np.full(4, 37.0), rtol=0, atol=1e-9)


def test_token_200_is_read_through_table_position_12(golden_dir):
    g = _load(golden_dir, "block_tables.json")["token_200"]
    t, pos = g["token"], g["table_position"]
    L = 16 * (pos + 1)
    table = list(range(pos + 1))[::-1]                      # distinct physical ids
    kc = np.zeros((pos + 1, 1, 16, 4), dtype=np.float32)
    vc = np.zeros((pos + 1, 1, 16, 4), dtype=np.float32)
    kc[table[pos], 0, t % 16, :] = 60.0
    vc[table[pos], 0, t % 16, :] = 3.25
    got = oracle.paged_decode(np.ones((1, 1, 4), np.float32), kc, vc, np.array([table], np.int32),
                              np.array([L], np.int32), 1.0)
    np.testing.assert_allclose(got[0, 0], np.full(4, 3.25), rtol=1e-9, atol=1e-9)


def test_logical_to_physical_example(golden_dir):
    """Logical blocks 0, 1, 2 stored in physical blocks 7, 3, 12."""
    table = _load(golden_dir, "block_tables.json")["logical_to_physical"]["table"]
    NB, L = 13, 40
    rng = np.random.default_rng(8)
    ck = [rng.standard_normal((1, L, 8)).astype(np.float32)]
    cv = [rng.standard_normal((1, L, 8)).astype(np.float32)]
    kc, vc = _scatter(ck, cv, [table], [L], NB)
    assert np.array_equal(kc[3, 0, :16], ck[0][0, 16:32])    # logical block 1 -> physical 3
    q = rng.standard_normal((1, 1, 8)).astype(np.float32)
    got = oracle.paged_decode(q, kc, vc, np.array([table], np.int32), np.array([L], np.int32), 0.35)
    np.testing.assert_allclose(got[0], _sdpa(q[0], ck[0], cv[0], 0.35, 1), rtol=1e-11, atol=1e-12)


def test_permuting_physical_blocks_changes_nothing():
    """Paging only changes addressing: moving blocks and remapping tables is bit-identical."""
    rng = np.random.default_rng(9)
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 4, 8, 2, 64, [3, 16, 45, 200], spare=5)
    ref = oracle.paged_decode(q, kc, vc, tables, L, 0.125)
    perm = rng.permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    got = oracle.paged_decode(q, kc2, vc2, t2, L, 0.125)
    assert np.array_equal(got, ref)


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(10)
    g = 4
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 3, 8, 2, 64, [5, 40, 90])
    got = oracle.paged_decode(q, kc, vc, tables, L, 0.125)
    kc_rep = np.repeat(kc, g, axis=1)
    vc_rep = np.repeat(vc, g, axis=1)
    ref = oracle.paged_decode(q, kc_rep, vc_rep, tables, L, 0.125)
    assert np.array_equal(got, ref)
    # and the group really matters: a wrong head mapping gives another answer
    assert not np.allclose(got[:, 1], got[:, 4])


def test_selected_pairs_match_full_output():
    rng = np.random.default_rng(11)
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 3, 4, 2, 32, [10, 20, 30])
    full = oracle.paged_decode(q, kc, vc, tables, L, 0.2, threads=2)
    sel = np.array([[2, 3], [0, 0], [1, 2]])
    part = oracle.paged_decode(q, kc, vc, tables, L, 0.2, sel=sel)
    for i, (b, h) in enumerate(sel):
        assert np.array_equal(part[i], full[b, h])


def test_empty_context_gives_zeros():
    rng = np.random.default_rng(12)
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 2, 2, 2, 16, [0, 5])
    got = oracle.paged_decode(q, kc, vc, tables, L, 1.0)
    assert np.array_equal(got[0], np.zeros((2, 16)))


def test_rejects_out_of_range_table_entry():
    rng = np.random.default_rng(13)
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 1, 1, 1, 16, [20])
    bad = tables.copy()
    bad[0, 1] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle.paged_decode(q, kc, vc, bad, L, 1.0)


# ---------------------------------------------------------------------------
# cache write and block copy
# ---------------------------------------------------------------------------

def test_cache_write_places_each_row_in_its_slot_and_nothing_else():
    wl = W.make_workload("tiny")
    hv = W.host_values(wl, poison_unused=False)
    kc, vc = hv.key_cache.copy(), hv.value_cache.copy()
    slots = wl.slot_mapping.copy()
    slots[1] = -1                                            # padding entry: no write
    oracle.cache_write(kc, vc, hv.key_new, hv.value_new, slots)
    changed = np.argwhere(np.any(kc != hv.key_cache, axis=-1))
    expect = {(int(s) // 16, h, int(s) % 16) for i, s in enumerate(slots) if s >= 0
              for h in range(wl.num_kv_heads)}
    assert {tuple(x) for x in changed} == expect
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(kc[s // 16, :, s % 16, :], hv.key_new[i])
        assert np.array_equal(vc[s // 16, :, s % 16, :], hv.value_new[i])


def test_cache_write_then_decode_sees_the_new_token():
    """After the write at position L, a dominant key on the new token returns its value."""
    wl = W.make_workload("tiny")
    hv = W.host_values(wl)
    kc, vc = hv.key_cache.copy(), hv.value_cache.copy()
    q = hv.query.copy()
    kn = np.zeros_like(hv.key_new)
    for b in range(wl.num_seqs):
        for h in range(wl.num_kv_heads):
            kn[b, h] = 80.0 * q[b, h] / np.linalg.norm(q[b, h])
    oracle.cache_write(kc, vc, kn, hv.value_new, wl.slot_mapping)
    got = oracle.paged_decode(q, kc, vc, wl.block_tables, wl.step_context_lens, 1.0)
    np.testing.assert_allclose(got, hv.value_new.astype(np.float64), rtol=1e-9, atol=1e-9)


def test_cache_write_rejects_slot_past_the_pool():
    wl = W.make_workload("tiny")
    hv = W.host_values(wl, poison_unused=False)
    bad = wl.slot_mapping.copy()
    bad[0] = wl.num_blocks * 16
    with pytest.raises(ValueError):
        oracle.cache_write(hv.key_cache, hv.value_cache, hv.key_new, hv.value_new, bad)


def test_block_copy_duplicates_whole_blocks_and_cow_is_invisible_to_decode():
    wl = W.make_workload("tiny")
    hv = W.host_values(wl, poison_unused=False)
    kc, vc = hv.key_cache.copy(), hv.value_cache.copy()
    tables = wl.block_tables.copy()
    free = sorted(set(range(wl.num_blocks)) - set(tables[tables >= 0].tolist()))
    pairs = np.array([[tables[2, 1], free[0]], [tables[3, 0], free[1]]], dtype=np.int32)
    before = oracle.paged_decode(hv.query, kc, vc, tables, wl.context_lens, wl.scale)
    oracle.block_copy(kc, vc, pairs)
    for s, d in pairs:
        assert np.array_equal(kc[d], kc[s]) and np.array_equal(vc[d], vc[s])
    untouched = [i for i in range(wl.num_blocks) if i not in set(pairs[:, 1].tolist())]
    assert np.array_equal(kc[untouched], hv.key_cache[untouched])
    tables[2, 1], tables[3, 0] = pairs[0, 1], pairs[1, 1]   # re-point to the copies
    after = oracle.paged_decode(hv.query, kc, vc, tables, wl.context_lens, wl.scale)
    assert np.array_equal(before, after)


# Block copy lists ("PagedAttention por dentro", "Copy-on-write para sampling
# paralelo"): every copy on the pages goes into a freshly taken block, so the
# pairs of one list are independent copies.  A pair whose destination another
# pair reads or writes is not such a copy and is skipped; the expectations
# below are written from the pools before the call.
def _numbered_pools(nb=6):
    kc = np.arange(nb * 2 * 16 * 2, dtype=np.float32).reshape(nb, 2, 16, 2)
    return kc, -kc - 1.0


def test_block_copy_chained_list_skips_the_pair_that_overwrites_a_source():
    kc, vc = _numbered_pools()
    k0, v0 = kc.copy(), vc.copy()
    skipped = oracle.block_copy(kc, vc, [[0, 1], [1, 2], [3, 4]])
    assert skipped
    # (0, 1) would overwrite the source of (1, 2): skipped; (1, 2) copies the old block 1
    assert np.array_equal(kc[1], k0[1]) and np.array_equal(vc[1], v0[1])
    assert np.array_equal(kc[2], k0[1]) and np.array_equal(vc[2], v0[1])
    assert np.array_equal(kc[4], k0[3]) and np.array_equal(vc[4], v0[3])
    for b in (0, 3, 5):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])


def test_block_copy_duplicate_destination_skips_both_pairs():
    kc, vc = _numbered_pools()
    k0, v0 = kc.copy(), vc.copy()
    assert oracle.block_copy(kc, vc, [[0, 2], [1, 2], [0, 5]])
    assert np.array_equal(kc[2], k0[2]) and np.array_equal(vc[2], v0[2])
    assert np.array_equal(kc[5], k0[0]) and np.array_equal(vc[5], v0[0])
    # two copies of one source into distinct fresh blocks are independent
    kc, vc = _numbered_pools()
    assert not oracle.block_copy(kc, vc, [[0, 1], [0, 2]])
    assert np.array_equal(kc[1], k0[0]) and np.array_equal(kc[2], k0[0])


def test_block_copy_self_pair_is_a_no_op_that_blocks_nothing():
    kc, vc = _numbered_pools()
    k0, v0 = kc.copy(), vc.copy()
    assert not oracle.block_copy(kc, vc, [[3, 3], [3, 1]])
    assert np.array_equal(kc[3], k0[3]) and np.array_equal(kc[1], k0[3])
    assert np.array_equal(vc[1], v0[3])


def test_block_copy_skips_pairs_outside_the_pool():
    kc, vc = _numbered_pools()
    k0 = kc.copy()
    assert oracle.block_copy(kc, vc, [[0, 6], [-1, 2], [4, 5]])
    assert np.array_equal(kc[:5], k0[:5]) and np.array_equal(kc[5], k0[4])


# ---------------------------------------------------------------------------
# sliding window ("PagedAttention por dentro", "Sliding window attention")
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("window", [1, 5, 16, 17, 64])
def test_window_matches_library_attention_on_the_last_tokens(window):
    rng = np.random.default_rng(50 + window)
    lens = [3, 16, 40, 130]
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 4, 8, 2, 64, lens)
    got = oracle.paged_decode(q, kc, vc, tables, L, 0.2, window=window)
    for b, n in enumerate(lens):
        lo = max(0, n - window)
        want = _sdpa(q[b], ck[b][:, lo:], cv[b][:, lo:], 0.2, 4)
        np.testing.assert_allclose(got[b], want, rtol=1e-11, atol=1e-12)


def test_window_of_one_returns_the_last_value_and_wide_windows_change_nothing():
    rng = np.random.default_rng(60)
    lens = [7, 33]
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 2, 4, 4, 32, lens)
    one = oracle.paged_decode(q, kc, vc, tables, L, 0.5, window=1)
    for b, n in enumerate(lens):
        assert np.array_equal(one[b], cv[b][:, n - 1, :].astype(np.float64))
    full = oracle.paged_decode(q, kc, vc, tables, L, 0.5)
    assert np.array_equal(oracle.paged_decode(q, kc, vc, tables, L, 0.5, window=33), full)
    assert np.array_equal(oracle.paged_decode(q, kc, vc, tables, L, 0.5, window=1000), full)


def test_window_never_reads_released_blocks():
    """Blocks wholly before the window may be gone (table entry -1)."""
    rng = np.random.default_rng(61)
    lens = [100]
    q, ck, cv, kc, vc, tables, L = _random_paged(rng, 1, 2, 2, 16, lens)
    want = oracle.paged_decode(q, kc, vc, tables, L, 0.3, window=40)
    t2 = tables.copy()
    t2[0, :3] = -1                       # positions 0..47 released; window starts at 60
    got = oracle.paged_decode(q, kc, vc, t2, L, 0.3, window=40)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# Chunked prefill
# ---------------------------------------------------------------------------
def _random_chunks(rng, Hq, Hkv, D, specs, spare=3):
    """specs: (cached tokens C, chunk tokens T) per sequence; context L = C + T."""
    lens = [c + t for c, t in specs]
    _, ck, cv, kc, vc, tables, L = _random_paged(rng, len(specs), Hq, Hkv, D, lens, spare)
    qs = np.zeros(len(specs) + 1, dtype=np.int32)
    qs[1:] = np.cumsum([t for _, t in specs])
    q = rng.standard_normal((int(qs[-1]), Hq, D)).astype(np.float32)
    return q, ck, cv, kc, vc, tables, L, qs


def _sdpa_causal(q, ck, cv, scale, group, cached, window=0):
    """Library attention of T query rows at positions cached .. cached+T-1 over
    contiguous K/V [Hkv][L][D], with an explicit causal (and window) mask."""
    T, L = q.shape[0], ck.shape[1]
    i = np.arange(T)[:, None] + cached
    j = np.arange(L)[None, :]
    allowed = j <= i
    if window:
        allowed &= j > i - window
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]   # [1,Hq,T,D]
    kt = torch.from_numpy(ck.astype(np.float64))[None]
    vt = torch.from_numpy(cv.astype(np.float64))[None]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(allowed), scale=scale, enable_gqa=group > 1)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("B,Hq,Hkv,D,specs", [
    (2, 8, 2, 64, [(0, 21), (37, 19), (100, 1)]),
    (1, 4, 4, 32, [(0, 50)]),
    (2, 16, 2, 128, [(15, 17), (48, 33)]),
])
def test_prefill_matches_library_causal_attention(B, Hq, Hkv, D, specs):
    rng = np.random.default_rng(70 + Hq + D)
    q, ck, cv, kc, vc, tables, L, qs = _random_chunks(rng, Hq, Hkv, D, specs)
    got = oracle.paged_prefill(q, kc, vc, tables, L, qs, 0.15)
    for b, (c, t) in enumerate(specs):
        want = _sdpa_causal(q[qs[b]:qs[b + 1]], ck[b], cv[b], 0.15, Hq // Hkv, c)
        np.testing.assert_allclose(got[qs[b]:qs[b + 1]], want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("window", [1, 9, 40])
def test_prefill_window_matches_library_attention(window):
    rng = np.random.default_rng(80 + window)
    specs = [(0, 30), (25, 20), (64, 3)]
    q, ck, cv, kc, vc, tables, L, qs = _random_chunks(rng, 8, 4, 64, specs)
    got = oracle.paged_prefill(q, kc, vc, tables, L, qs, 0.3, window=window)
    for b, (c, t) in enumerate(specs):
        want = _sdpa_causal(q[qs[b]:qs[b + 1]], ck[b], cv[b], 0.3, 2, c, window)
        np.testing.assert_allclose(got[qs[b]:qs[b + 1]], want, rtol=1e-11, atol=1e-12)


def test_prefill_first_row_of_a_fresh_sequence_is_its_own_value():
    """Position 0 attends to itself alone: softmax weight 1."""
    rng = np.random.default_rng(90)
    q, ck, cv, kc, vc, tables, L, qs = _random_chunks(rng, 4, 2, 32, [(0, 5), (0, 1)])
    got = oracle.paged_prefill(q, kc, vc, tables, L, qs, 0.5)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(got[qs[b], h], cv[b][h // 2, 0].astype(np.float64))


def test_prefill_rows_equal_decode_and_chunking_changes_nothing():
    """Row i of a chunk is the decode of that query over the first C + i + 1
    positions, and splitting one prompt into chunks gives the same rows."""
    rng = np.random.default_rng(91)
    q, ck, cv, kc, vc, tables, L, qs = _random_chunks(rng, 8, 2, 64, [(0, 70)])
    whole = oracle.paged_prefill(q, kc, vc, tables, L, qs, 0.2)
    for i in (0, 15, 16, 69):
        dec = oracle.paged_decode(q[i:i + 1], kc, vc, tables, np.array([i + 1], np.int32), 0.2)
        assert np.array_equal(dec[0], whole[i])
    for cut in (1, 16, 33):
        a = oracle.paged_prefill(q[:cut], kc, vc, tables, np.array([cut], np.int32),
                                 np.array([0, cut], np.int32), 0.2)
        b = oracle.paged_prefill(q[cut:], kc, vc, tables, L, np.array([0, 70 - cut], np.int32),
                                 0.2)
        assert np.array_equal(np.concatenate([a, b]), whole)
