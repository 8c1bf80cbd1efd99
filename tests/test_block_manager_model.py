"""Pins for the block-manager model (host logic; no GPU)."""
import json
import os
import random

import pytest

from oracle.block_manager_model import BlockManagerModel, NoBlocks


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "block_tables.json")) as f:
        return json.load(f)


def test_273_tokens_take_18_blocks(golden_dir):
    g = _golden(golden_dir)["tokens_to_blocks"]
    bm = BlockManagerModel(64)
    assert len(bm.alloc_seq(0, g["tokens"])) == g["blocks"]
    bm.check()


def test_273_token_session_wastes_15_of_288_slots(golden_dir):
    """Internal fragmentation of the pages' 273-token session: 18 blocks of 16
    reserve 288 slots, 273 hold a token, so 15 / 288 (5.2 %) of the reservation is
    waste ("Cómo funciona realmente vLLM", "La sobre-reserva estática y los tres
    tipos de desperdicio": internal fragmentation is reserved slots that are never
    written)."""
    g = _golden(golden_dir)["tokens_to_blocks"]
    bm = BlockManagerModel(64)
    bm.alloc_seq(0, g["tokens"])
    st = bm.stats()
    assert st["used_blocks"] == g["blocks"] and st["reserved_slots"] == 288
    assert st["filled_slots"] == g["tokens"] and st["logical_tokens"] == g["tokens"]
    assert st["internal_fragmentation"] == pytest.approx(15 / 288, abs=0, rel=1e-15)
    assert st["free_blocks"] == 64 - 18 and st["shared_blocks"] == 0


def test_forked_sessions_share_slots_until_they_diverge():
    """A fork shares every block: logical tokens double, filled slots do not.
    Its first new token copies the shared last block (8 tokens) into a fresh one."""
    bm = BlockManagerModel(16)
    bm.alloc_seq(0, 40)                                # 3 blocks: 16 + 16 + 8
    bm.fork(0, 1)
    st = bm.stats()
    assert (st["used_blocks"], st["shared_blocks"], st["filled_slots"], st["logical_tokens"]) == (3, 3, 40, 80)
    _, cow = bm.append_slot(1)                         # token 40 of the child
    assert cow is not None
    st = bm.stats()
    assert (st["used_blocks"], st["shared_blocks"]) == (4, 2)
    assert st["filled_slots"] == 16 + 16 + 8 + 9 and st["logical_tokens"] == 81
    assert st["internal_fragmentation"] == pytest.approx((64 - 49) / 64, rel=1e-15)


def test_waste_of_the_7b_shaped_batch_is_under_four_percent():
    """The pages' figure for paging ("PagedAttention por dentro", opening section:
    under 4 % waste) holds for the 64 contexts of the 7B-shaped decode batch
    (lengths uniform in [128, 2048]): only each last block can be partly empty."""
    import workloads as W
    wl = W.make_workload("llama7b_mha")
    bm = BlockManagerModel(wl.num_blocks)
    for b, L in enumerate(wl.context_lens):
        bm.alloc_seq(b, int(L))
    st = bm.stats()
    assert st["filled_slots"] == int(wl.context_lens.sum())
    assert 0 < st["internal_fragmentation"] < 0.04


def test_128_tokens_on_32_layers_take_256_blocks(golden_dir):
    """One pool per layer: a session holds blocks in each of the 32 layers' pools."""
    g = _golden(golden_dir)["blocks_per_session_all_layers"]
    pools = [BlockManagerModel(16) for _ in range(g["layers"])]
    total = sum(len(p.alloc_seq(0, g["tokens"])) for p in pools)
    assert total == g["blocks"]


def test_growth_rule_allocates_only_on_block_boundaries():
    """Token N goes to the last block when N mod 16 != 0, else to a newly appended block."""
    bm = BlockManagerModel(8)
    bm.alloc_seq(0, 0)
    for n in range(64):
        before = len(bm.table(0))
        slot, cow = bm.append_slot(0)
        assert cow is None
        grew = len(bm.table(0)) - before
        assert grew == (1 if n % 16 == 0 else 0)
        assert slot == bm.table(0)[n // 16] * 16 + n % 16
    assert bm.num_free() == 4
    bm.check()


def test_fork_shares_and_append_copies_only_the_last_block():
    bm = BlockManagerModel(10)
    bm.alloc_seq(0, 40)                  # 3 blocks, last one holds 8 tokens
    bm.fork(0, 1)
    assert bm.table(1) == bm.table(0)
    assert all(bm.ref_count(b) == 2 for b in bm.table(0))
    slot, cow = bm.append_slot(1)        # divergence inside the shared last block
    src, dst = cow
    assert src == bm.table(0)[2] and dst == bm.table(1)[2] and src != dst
    assert bm.table(1)[:2] == bm.table(0)[:2]
    assert slot == dst * 16 + 8
    assert bm.ref_count(src) == 1 and bm.ref_count(dst) == 1
    # the parent now owns its last block alone: no copy for it
    _, cow0 = bm.append_slot(0)
    assert cow0 is None
    bm.check()


def test_fork_at_block_boundary_needs_no_copy():
    bm = BlockManagerModel(10)
    bm.alloc_seq(0, 32)
    bm.fork(0, 1)
    _, cow = bm.append_slot(1)
    assert cow is None
    assert bm.table(1)[:2] == bm.table(0)
    bm.check()


def test_free_returns_blocks_and_lifo_reuse():
    bm = BlockManagerModel(6)
    t0 = bm.alloc_seq(0, 33)             # 0, 1, 2
    assert t0 == [0, 1, 2]
    bm.alloc_seq(1, 16)                  # 3
    bm.free_seq(0)
    assert bm.num_free() == 5
    assert bm.alloc_seq(2, 20) == [0, 1]
    bm.check()


def test_exhaustion_changes_nothing():
    bm = BlockManagerModel(3)
    bm.alloc_seq(0, 32)
    with pytest.raises(NoBlocks):
        bm.alloc_seq(1, 20)
    assert 1 not in bm.tables and bm.num_free() == 1
    bm.alloc_seq(1, 16)
    with pytest.raises(NoBlocks):
        bm.append_slot(1)
    assert bm.num_tokens(1) == 16
    bm.check()


def test_random_operations_keep_invariants():
    rng = random.Random(5)
    bm = BlockManagerModel(40)
    live = []
    nxt = 0
    for _ in range(3000):
        op = rng.random()
        try:
            if op < 0.2 or not live:
                bm.alloc_seq(nxt, rng.randrange(0, 70))
                live.append(nxt)
                nxt += 1
            elif op < 0.35:
                bm.fork(rng.choice(live), nxt)
                live.append(nxt)
                nxt += 1
            elif op < 0.85:
                bm.append_slot(rng.choice(live))
            else:
                s = rng.choice(live)
                bm.free_seq(s)
                live.remove(s)
        except NoBlocks:
            pass
        bm.check()
    for s in list(live):
        bm.free_seq(s)
    assert bm.num_free() == 40
