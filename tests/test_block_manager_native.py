"""The native (C++) block manager against the Python model, step by step (CPU only)."""
import random

import numpy as np
import pytest

import paged_kv_cache_100_gb300 as pkv
from oracle.block_manager_model import BlockManagerModel, NoBlocks
from paged_kv_cache_100_gb300.build import build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _same(bm, model, live):
    assert bm.stats() == model.stats()
    assert bm.num_free() == model.num_free()
    for s in live:
        assert bm.table(s) == model.table(s)
        assert bm.num_tokens(s) == model.num_tokens(s)
    for b in range(model.num_blocks):
        assert bm.ref_count(b) == model.ref_count(b)


def test_random_operations_match_the_model():
    rng = random.Random(11)
    bm, model = pkv.BlockManager(48), BlockManagerModel(48)
    live, nxt = [], 0
    for step in range(4000):
        op = rng.random()
        if op < 0.15 or not live:
            n = rng.randrange(0, 90)
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
        elif op < 0.3:
            p = rng.choice(live)
            model.fork(p, nxt)
            bm.fork(p, nxt)
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
        elif op < 0.88:
            s = rng.choice(live)
            j = rng.randrange(0, max(1, len(model.table(s))))
            if model.table(s):
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
        if step % 50 == 0:
            _same(bm, model, live)
    _same(bm, model, live)


def test_batch_step_and_dense_tables():
    bm, model = pkv.BlockManager(64), BlockManagerModel(64)
    for s, n in enumerate([0, 15, 16, 33]):
        bm.alloc_seq(s, n)
        model.alloc_seq(s, n)
    bm.fork(3, 4)
    model.fork(3, 4)
    seqs = [0, 1, 2, 3, 4]
    slots, pairs = bm.append_slots(seqs)
    want = [model.append_slot(s) for s in seqs]
    assert list(slots) == [w[0] for w in want]
    assert [tuple(p) for p in pairs] == [w[1] for w in want if w[1] is not None]
    tables, lens = bm.fill_tables(seqs, 6)
    for i, s in enumerate(seqs):
        t = model.table(s)
        assert list(tables[i, :len(t)]) == t and np.all(tables[i, len(t):] == -1)
        assert lens[i] == model.num_tokens(s)


def test_unknown_and_duplicate_sequences():
    bm = pkv.BlockManager(4)
    bm.alloc_seq(1, 5)
    with pytest.raises(pkv.PagedKVError):
        bm.alloc_seq(1, 5)
    with pytest.raises(pkv.PagedKVError):
        bm.free_seq(2)
    with pytest.raises(pkv.PagedKVError):
        bm.fork(7, 8)
    with pytest.raises(KeyError):
        bm.table(9)
