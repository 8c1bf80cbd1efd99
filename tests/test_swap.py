"""Swap (preemption to host memory) on the CPU: the oracle's swap against the
pool's own contents and against decode, the block-manager model's scenario, and
the native manager against the model."""
import random

import numpy as np
import pytest

import oracle
import paged_kv_cache_100_gb300 as pkv
import workloads as W
from oracle.block_manager_model import BlockManagerModel, NoBlocks
from paged_kv_cache_100_gb300.build import build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def test_oracle_swap_round_trip_to_other_blocks_keeps_decode_bit_identical():
    """Moving a sequence's blocks out and back into different physical blocks, with
    its table remapped, changes nothing the decode sees (paging only changes
    addressing)."""
    wl = W.custom_workload(3, 4, 2, 64, [37, 80, 5], dtype="bf16", spare_blocks=12, seed=4)
    hv = W.host_values(wl)
    lens = np.asarray(wl.context_lens, np.int32)
    before = oracle.paged_decode(hv.query, hv.key_cache, hv.value_cache, wl.block_tables, lens,
                                 wl.scale)
    kc, vc = hv.key_cache.copy(), hv.value_cache.copy()
    nb1 = -(-int(lens[1]) // 16)
    ids = wl.block_tables[1, :nb1].copy()
    staging = oracle.swap_out(kc, vc, ids)
    assert staging.shape == (nb1, 2, 2, 16, 64)
    for i, b in enumerate(ids):                       # staging order = table order
        assert np.array_equal(staging[i, 0], hv.key_cache[b])
        assert np.array_equal(staging[i, 1], hv.value_cache[b])
    kc[ids] = 0x7FC0                                  # the blocks get reused and overwritten
    vc[ids] = 0x7FC0
    used = set(wl.block_tables[wl.block_tables >= 0].tolist())
    spare = [b for b in range(wl.num_blocks) if b not in used][:nb1]
    oracle.swap_in(kc, vc, spare, staging)
    tables = wl.block_tables.copy()
    tables[1, :nb1] = spare
    after = oracle.paged_decode(hv.query, kc, vc, tables, lens, wl.scale)
    assert np.array_equal(before.view(np.uint64), after.view(np.uint64))


def test_oracle_swap_in_rejects_repeated_ids():
    kc = np.zeros((4, 1, 16, 16), np.float32)
    with pytest.raises(ValueError):
        oracle.swap_in(kc, kc.copy(), [1, 1], np.zeros((2, 2, 1, 16, 16), np.float32))


def test_model_swap_scenario():
    bm = BlockManagerModel(8)
    bm.alloc_seq(0, 40)                               # blocks 0, 1, 2
    bm.alloc_seq(1, 20)                               # blocks 3, 4
    assert bm.swap_out(0) == [0, 1, 2]
    assert bm.table(0) == [-2, -2, -2] and bm.num_free() == 6
    with pytest.raises(ValueError):
        bm.append_slot(0)
    bm.alloc_seq(2, 48)                               # reuses 0, 1, 2 (freed last first)
    assert bm.table(2) == [0, 1, 2]
    assert bm.swap_in(0) == [5, 6, 7]
    assert bm.table(0) == [5, 6, 7] and bm.num_free() == 0
    slot, cow = bm.append_slot(0)
    assert slot == 7 * 16 + 8 and cow is None
    bm.check()


def test_model_swap_of_shared_and_trimmed_tables():
    bm = BlockManagerModel(8)
    bm.alloc_seq(0, 50)                               # 0, 1, 2, 3
    bm.fork(0, 1)
    bm.trim_window(1, 10)                             # window [40, 50): drops blocks 0, 1
    assert bm.table(1) == [-1, -1, 2, 3]
    assert bm.swap_out(1) == [2, 3]
    assert bm.table(1) == [-1, -1, -2, -2]
    assert [bm.ref_count(b) for b in range(4)] == [1, 1, 1, 1]
    with pytest.raises(NoBlocks):
        _full_swap_in(bm)                             # all or nothing
    assert bm.table(1) == [-1, -1, -2, -2]
    bm.free_seq(0)                                    # releases 3, 2, 1, 0: 0 is on top
    assert bm.swap_in(1) == [0, 1]                    # private copies now
    assert bm.table(1) == [-1, -1, 0, 1]
    bm.check()


def _full_swap_in(bm):
    bm.alloc_seq(9, 16 * bm.num_free())               # exhaust the pool
    try:
        bm.swap_in(1)
    finally:
        bm.free_seq(9)


def test_native_swap_matches_the_model():
    rng = random.Random(23)
    bm, model = pkv.BlockManager(40), BlockManagerModel(40)
    live, out, nxt = [], [], 0
    for step in range(4000):
        op = rng.random()
        if op < 0.12 or not (live or out):
            n = rng.randrange(0, 100)
            try:
                model.alloc_seq(nxt, n)
                bm.alloc_seq(nxt, n)
                live.append(nxt)
            except NoBlocks:
                with pytest.raises(pkv.PagedKVError):
                    bm.alloc_seq(nxt, n)
            nxt += 1
        elif op < 0.25 and live:
            s = rng.choice(live)
            assert bm.swap_out(s) == model.swap_out(s)
            live.remove(s)
            out.append(s)
        elif op < 0.38 and out:
            s = rng.choice(out)
            try:
                want = model.swap_in(s)
            except NoBlocks:
                want = None
            if want is None:
                with pytest.raises(pkv.PagedKVError):
                    bm.swap_in(s)
            else:
                assert bm.swap_in(s) == want
                out.remove(s)
                live.append(s)
        elif op < 0.48 and live:
            s, w = rng.choice(live), rng.randrange(1, 60)
            assert bm.trim_window(s, w) == model.trim_window(s, w)
        elif op < 0.56 and live:
            s = rng.choice(live)
            model.fork(s, nxt)
            bm.fork(s, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.85 and live:
            s = rng.choice(live)
            try:
                want = model.append_slot(s)
            except NoBlocks:
                want = None
            if want is None:
                with pytest.raises(pkv.PagedKVError):
                    bm.append_slot(s)
            else:
                assert bm.append_slot(s) == want
        elif out and rng.random() < 0.5:
            s = rng.choice(out)
            with pytest.raises(pkv.PagedKVError):
                bm.append_slot(s)                     # a swapped sequence cannot grow
            model.free_seq(s)
            bm.free_seq(s)
            out.remove(s)
        elif live:
            s = rng.choice(live)
            model.free_seq(s)
            bm.free_seq(s)
            live.remove(s)
        if step % 25 == 0:
            model.check()
            assert bm.stats() == model.stats()
            assert bm.num_free() == model.num_free()
            for s in live + out:
                assert bm.table(s) == model.table(s)
            for b in range(40):
                assert bm.ref_count(b) == model.ref_count(b)
