"""The KV byte accounting behind the bench's roofline, pinned to the sizes the pages
print (tests/golden/kv_bytes.json, each entry citing its page and section).

The formula ("KV cache: la memoria de trabajo que sostiene la inferencia LLM",
"El precio: cuánto pesa la mochila"): K and V of every token, 2 · layers · KV heads ·
head_dim · bytes per element.  A decode layer of the bench moves that per attended
token for one layer, plus Q, O and the table entries."""
import json
import os

import numpy as np
import pytest

import bench
import workloads as W


@pytest.fixture(scope="module")
def golden(golden_dir):
    with open(os.path.join(golden_dir, "kv_bytes.json")) as f:
        return json.load(f)


def test_bytes_per_token_table(golden):
    t = golden["per_token_table"]
    for row in t["rows"]:
        per_token = bench.kv_bytes_per_token(row["n_layers"], row["n_kv_heads"], row["head_dim"],
                                             t["bytes_per_elem"])
        assert per_token == row["bytes_per_token"], row["model"]
        for key, ctx in (("gb_8k", 8192), ("gb_32k", 32768), ("gb_128k", 131072)):
            assert round(per_token * ctx / 2**30, 2) == row[key], (row["model"], key)


def test_70b_prompt_of_4096_tokens(golden):
    g = golden["prompt_70b"]
    per_token = bench.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"],
                                         g["bytes_per_elem"])
    assert per_token == g["bytes_per_token"]
    assert round(per_token * g["tokens"] / 1e9, 2) == g["gb_decimal"]


def test_one_block_of_all_layers(golden):
    g = golden["block_bytes"]
    block = g["block_size"] * bench.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"],
                                                       g["head_dim"], g["bytes_per_elem"])
    assert block == g["mb"] * 2**20


def test_decode_layer_bytes_are_the_formula_for_one_layer(golden):
    """One sequence of the 70B-shaped prompt through one decode layer: the K/V term
    of the bench's algorithmic bytes is the pages' 1.34 GB over 80 layers."""
    g = golden["prompt_70b"]
    wl = W.custom_workload(1, 64, g["n_kv_heads"], g["head_dim"], [g["tokens"]], dtype="bf16")
    b = bench.decode_algorithmic_bytes(wl, lens=[g["tokens"]])
    assert b["kv"] * g["n_layers"] == g["bytes_per_token"] * g["tokens"]
    assert b["q"] == b["o"] == 64 * g["head_dim"] * 2
    assert b["tables"] == 4 * (g["tokens"] // 16) + 4
    assert b["total"] == b["kv"] + b["q"] + b["o"] + b["tables"]


def test_window_counts_only_attended_positions():
    wl = W.custom_workload(3, 8, 2, 128, [10, 100, 5000], dtype="bf16")
    full = bench.decode_algorithmic_bytes(wl, lens=[10, 100, 5000])
    win = bench.decode_algorithmic_bytes(wl, lens=[10, 100, 5000], window=64)
    per_row = bench.kv_bytes_per_token(1, 2, 128, 2)
    assert full["kv"] == (10 + 100 + 5000) * per_row
    assert win["kv"] == (10 + 64 + 64) * per_row


def test_unique_bytes_count_a_shared_block_once():
    """Two sequences whose tables share their first block: the shared slots count once."""
    wl = W.custom_workload(2, 4, 4, 64, [40, 40], dtype="bf16")
    wl.block_tables[1, 0] = wl.block_tables[0, 0]
    lens = np.asarray([40, 40])
    per_row = bench.kv_bytes_per_token(1, 4, 64, 2)
    assert bench.unique_kv_bytes(wl, lens=lens) == (80 - 16) * per_row
    assert bench.decode_algorithmic_bytes(wl, lens=lens)["kv"] == 80 * per_row


def test_causal_pair_count_is_the_pages_cost_table(golden_dir):
    """The prefill roofline counts (query row, attended position) pairs.  A fresh
    prompt of N tokens (nothing cached) has N(N+1)/2 of them: the "without a KV
    cache" column of the pages' cost table, where step i attends i tokens."""
    with open(os.path.join(golden_dir, "attention_cost.json")) as f:
        rows = json.load(f)["cost_table"]["rows"]
    for r in rows:
        n = r["tokens"]
        pw = W.PrefillWorkload("fresh", 1, 1, 1, 128, 1.0, np.zeros(1, np.int32),
                               np.asarray([n], np.int32), np.zeros((1, 1), np.int32), 1)
        pairs = bench.prefill_pairs(pw)
        assert pairs == r["without_cache"], n
        assert pairs // r["with_cache"] == r["ratio"], n
        # QK^T and PV: 2 * head_dim flops each per pair and head
        assert bench.prefill_flops(pw) == 4 * 128 * pairs
    # a window caps each row's pairs: the last W positions only
    pw = W.PrefillWorkload("fresh", 1, 1, 1, 128, 1.0, np.zeros(1, np.int32),
                           np.asarray([1024], np.int32), np.zeros((1, 1), np.int32), 1)
    assert bench.prefill_pairs(pw, window=128) == 8256 + (1024 - 128) * 128
