"""Prefix caching in the block manager (CPU): the model against published FNV-1a
vectors and worked scenarios, and the native manager against the model."""
import random

import numpy as np
import pytest

import paged_kv_cache_100_gb300 as pkv
from oracle.block_manager_model import BlockManagerModel, NoBlocks, block_keys, fnv1a64
from paged_kv_cache_100_gb300.build import build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def test_fnv1a64_published_vectors():
    # test vectors of the FNV-1a 64-bit hash
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_keys_chain_over_the_whole_prefix():
    a = list(range(48))
    b = list(range(16)) + [99] + list(range(17, 48))      # differs inside block 1
    ka, kb = block_keys(a), block_keys(b)
    assert len(ka) == 3 and ka[0] == kb[0]
    assert ka[1] != kb[1] and ka[2] != kb[2]              # block 2 differs through its parent


def test_same_system_prompt_reuses_blocks():
    """A request that begins like a finished one reuses its full blocks."""
    bm = BlockManagerModel(32)
    prompt_a = list(range(1000, 1100))                    # 100 tokens: 6 full blocks + 4
    assert bm.alloc_seq_cached(0, prompt_a) == 0
    assert bm.register_prefix(0, prompt_a) == 6
    table_a = bm.table(0)
    bm.free_seq(0)
    assert bm.num_evictable() == 6 and bm.num_free() == 26
    prompt_b = prompt_a[:80] + [7] * 30                   # same first 80 tokens
    assert bm.alloc_seq_cached(1, prompt_b) == 80
    assert bm.table(1)[:5] == table_a[:5]
    assert all(bm.ref_count(b) == 1 for b in table_a[:5])
    assert bm.alloc_seq_cached(2, [5] * 40) == 0          # unrelated prompt
    bm.check()


def test_evictable_blocks_are_reused_oldest_first_and_lose_their_key():
    bm = BlockManagerModel(4)
    for s, base in ((0, 0), (1, 100)):
        toks = list(range(base, base + 32))
        bm.alloc_seq_cached(s, toks)
        bm.register_prefix(s, toks)
    first = bm.table(0)
    bm.free_seq(0)                                        # released first: oldest
    bm.free_seq(1)
    assert bm.num_free() == 0 and bm.num_evictable() == 4
    bm.alloc_seq(2, 16)                                   # takes the oldest evictable block
    taken = bm.table(2)[0]
    assert taken == first[-1]                              # free_seq releases last entry first
    # seq 0's second block lost its key; its first block is still cached
    assert bm.alloc_seq_cached(3, list(range(0, 32))) == 16
    assert bm.table(3)[0] == first[0]
    bm.check()


def _random_tokens(rng, prompts):
    base = rng.choice(prompts)
    cut = rng.randrange(0, len(base) + 1)
    return base[:cut] + [rng.randrange(0, 8) for _ in range(rng.randrange(0, 40))]


def test_native_prefix_cache_matches_the_model():
    rng = random.Random(17)
    prompts = [[rng.randrange(0, 5) for _ in range(rng.randrange(16, 90))] for _ in range(4)]
    bm, model = pkv.BlockManager(60), BlockManagerModel(60)
    live, nxt, toks = [], 0, {}
    for step in range(3000):
        op = rng.random()
        if op < 0.25 or not live:
            t = _random_tokens(rng, prompts)
            try:
                want = model.alloc_seq_cached(nxt, t)
            except NoBlocks:
                want = None
            if want is None:
                with pytest.raises(pkv.PagedKVError):
                    bm.alloc_seq_cached(nxt, t)
            else:
                assert bm.alloc_seq_cached(nxt, t) == want
                live.append(nxt)
                toks[nxt] = t
            nxt += 1
        elif op < 0.45:
            s = rng.choice(live)
            assert bm.register_prefix(s, toks[s]) == model.register_prefix(s, toks[s])
        elif op < 0.6:
            s = rng.choice(live)
            model.fork(s, nxt)
            bm.fork(s, nxt)
            live.append(nxt)
            toks[nxt] = list(toks[s])
            nxt += 1
        elif op < 0.75:
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
                toks[s].append(rng.randrange(0, 8))
        elif op < 0.8:
            s = rng.choice(live)
            if model.table(s):
                j = rng.randrange(len(model.table(s)))
                try:
                    want = model.make_private(s, j)
                except NoBlocks:
                    want = "full"
                if want == "full":
                    with pytest.raises(pkv.PagedKVError):
                        bm.make_private(s, j)
                else:
                    assert bm.make_private(s, j) == want
        else:
            s = rng.choice(live)
            model.free_seq(s)
            bm.free_seq(s)
            live.remove(s)
        if step % 25 == 0:
            model.check()
            assert bm.stats() == model.stats()
            assert bm.num_free() == model.num_free()
            assert bm.num_evictable() == model.num_evictable()
            for s in live:
                assert bm.table(s) == model.table(s)
            for b in range(60):
                assert bm.ref_count(b) == model.ref_count(b)


def test_making_a_cached_block_private_drops_its_key():
    """A registered block about to be written in place (make_private on a block
    only its own sequence holds) must leave the prefix cache: a later sequence
    with the same tokens may not reuse it."""
    toks = list(range(40))
    for make in (BlockManagerModel, pkv.BlockManager):
        bm = make(16)
        assert bm.alloc_seq_cached(0, toks) == 0
        assert bm.register_prefix(0, toks) == 2
        assert bm.make_private(0, 1) is None          # private: written in place
        assert bm.alloc_seq_cached(1, toks) == 16     # block 0 reused, block 1 not
        assert bm.table(1)[0] == bm.table(0)[0] and bm.table(1)[1] != bm.table(0)[1]


def test_trim_window_releases_blocks_before_the_window():
    """Only blocks wholly before the last W tokens go back to the pool."""
    bm = BlockManagerModel(16)
    bm.alloc_seq(0, 70)                                   # blocks 0..4, positions 0..69
    assert bm.trim_window(0, 40) == 1                     # window [30, 70): block 0 ends at 15
    assert bm.table(0) == [-1, 1, 2, 3, 4]
    assert bm.trim_window(0, 40) == 0                     # idempotent
    assert bm.trim_window(0, 16) == 2                     # window [54, 70): blocks 1, 2 die
    assert bm.table(0) == [-1, -1, -1, 3, 4]
    assert bm.num_free() == 11 + 3
    assert bm.trim_window(0, 1000) == 0                   # window longer than the context
    slot, cow = bm.append_slot(0)                         # growth is unaffected
    assert slot == 4 * 16 + 6 and cow is None
    bm.fork(0, 1)
    assert [bm.ref_count(b) for b in (3, 4)] == [2, 2]
    with pytest.raises(ValueError):
        bm.make_private(1, 0)
    bm.free_seq(0)
    bm.free_seq(1)
    assert bm.num_free() == 16
    bm.check()


def test_native_sliding_window_matches_the_model():
    rng = random.Random(5)
    bm, model = pkv.BlockManager(48), BlockManagerModel(48)
    live, nxt = [], 0
    for step in range(3000):
        op = rng.random()
        if op < 0.15 or not live:
            n = rng.randrange(0, 120)
            try:
                model.alloc_seq(nxt, n)
                ok = True
            except NoBlocks:
                ok = False
            if ok:
                bm.alloc_seq(nxt, n)
                live.append(nxt)
            else:
                with pytest.raises(pkv.PagedKVError):
                    bm.alloc_seq(nxt, n)
            nxt += 1
        elif op < 0.35:
            s, w = rng.choice(live), rng.randrange(1, 80)
            assert bm.trim_window(s, w) == model.trim_window(s, w)
        elif op < 0.45:
            s = rng.choice(live)
            model.fork(s, nxt)
            bm.fork(s, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.8:
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
        else:
            s = rng.choice(live)
            model.free_seq(s)
            bm.free_seq(s)
            live.remove(s)
        if step % 25 == 0:
            model.check()
            assert bm.stats() == model.stats()
            assert bm.num_free() == model.num_free()
            for s in live:
                assert bm.table(s) == model.table(s)
            for b in range(48):
                assert bm.ref_count(b) == model.ref_count(b)
