"""GPU parity for chunked prefill: pa_prefill (tcgen05 tensor cores) through the C ABI
against the fp64 oracle.

Slots that hold no context token are NaN-poisoned, so a kernel that reads past a
context (or, with a window, before every row's window) shows it as NaN."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_100_gb300.build import build
    build()
    import paged_kv_cache_100_gb300 as m
    return m


def _case(hq, hkv, specs, seed, window=0):
    """specs: (cached C, chunk T) per sequence.  Returns host inputs for both sides."""
    lens = [c + t for c, t in specs]
    wl = W.custom_workload(len(specs), hq, hkv, D, lens, dtype="bf16", seed=seed)
    hv = W.host_values(wl)
    qs = np.zeros(len(specs) + 1, np.int32)
    qs[1:] = np.cumsum([t for _, t in specs])
    rng = np.random.default_rng(seed + 1000)
    q = W.to_bf16_bits(rng.standard_normal((int(qs[-1]), hq, D), dtype=np.float32))
    tables = wl.block_tables.copy()
    if window:
        # nothing before the first chunk row's window is needed: poison it and
        # drop the blocks wholly before it, as a block manager's trim would
        for b, (c, t) in enumerate(specs):
            lo = max(0, c + 1 - window)
            for pos in range(lo):
                phys = int(tables[b, pos // 16])
                hv.key_cache[phys, :, pos % 16] = 0x7FC0
                hv.value_cache[phys, :, pos % 16] = 0x7FC0
            tables[b, :lo // 16] = -1
    return wl, hv, q, qs, tables, np.asarray(lens, np.int32)


def _run(pkv, wl, hv, q, qs, tables, lens, window=0, max_query_len=None, scale=None):
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.prefill(H.host_to_device(q, torch.bfloat16),
                      H.host_to_device(hv.key_cache, torch.bfloat16),
                      H.host_to_device(hv.value_cache, torch.bfloat16),
                      torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                      torch.from_numpy(qs).cuda(), max_query_len,
                      wl.scale if scale is None else scale, window=window, status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


def _oracle(wl, hv, q, qs, tables, lens, window=0, scale=None):
    return oracle.paged_prefill(q, hv.key_cache, hv.value_cache, tables, lens, qs,
                                wl.scale if scale is None else scale, threads=8, window=window)


SPECS = [(0, 1), (0, 5), (0, 127), (0, 128), (0, 129), (17, 50), (300, 200), (1000, 31)]


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (8, 2), (16, 2), (16, 1)])
def test_prefill_matches_oracle(pkv, hq, hkv):
    wl, hv, q, qs, tables, lens = _case(hq, hkv, SPECS, seed=hq * 10 + hkv)
    got, st = _run(pkv, wl, hv, q, qs, tables, lens)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens), "bf16",
                   f"prefill {hq}/{hkv}")


@pytest.mark.parametrize("scale", [-0.0883883, -0.5, 0.0])
def test_prefill_nonpositive_scale(pkv, scale):
    """A negative scale reverses the order of the scores (the row maximum of
    scale * s sits at the smallest s); scale 0 weighs every attended position
    equally."""
    specs = [(0, 5), (0, 130), (300, 200), (17, 1)]
    wl, hv, q, qs, tables, lens = _case(8, 2, specs, seed=31)
    got, st = _run(pkv, wl, hv, q, qs, tables, lens, scale=scale)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens, scale=scale), "bf16",
                   f"prefill scale {scale}")


def test_long_fresh_prompt_spans_many_tiles(pkv):
    specs = [(0, 700), (0, 260)]
    wl, hv, q, qs, tables, lens = _case(8, 8, specs, seed=5)
    got, st = _run(pkv, wl, hv, q, qs, tables, lens)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens), "bf16", "long prompt")


@pytest.mark.parametrize("window", [1, 16, 100, 300])
def test_prefill_sliding_window_matches_oracle(pkv, window):
    specs = [(0, 64), (40, 90), (500, 140), (33, 1)]
    wl, hv, q, qs, tables, lens = _case(8, 2, specs, seed=window, window=window)
    got, st = _run(pkv, wl, hv, q, qs, tables, lens, window=window)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens, window), "bf16",
                   f"prefill window {window}")


def test_first_row_of_a_fresh_prompt_is_its_own_value(pkv):
    """Position 0 attends to itself alone: the output is that V row, rounded to bf16."""
    specs = [(0, 3), (0, 200)]
    wl, hv, q, qs, tables, lens = _case(8, 2, specs, seed=21)
    got, st = _run(pkv, wl, hv, q, qs, tables, lens)
    bits = H.device_to_host_bits(got)
    for b in range(2):
        phys = int(tables[b, 0])
        for h in range(8):
            assert np.array_equal(bits[qs[b], h], hv.value_cache[phys, h // 4, 0])


def test_chunked_equals_whole_prompt(pkv):
    """A prompt prefilled in two chunks gives the rows of the one-chunk prefill."""
    import torch
    wl, hv, q, qs, tables, lens = _case(8, 2, [(0, 300)], seed=31)
    whole, _ = _run(pkv, wl, hv, q, qs, tables, lens)
    cut = 137
    first, _ = _run(pkv, wl, hv, q[:cut], np.array([0, cut], np.int32), tables,
                    np.array([cut], np.int32))
    second, _ = _run(pkv, wl, hv, q[cut:], np.array([0, 300 - cut], np.int32), tables, lens)
    both = torch.cat([first, second])
    ref = _oracle(wl, hv, q, qs, tables, lens)
    H.assert_close(H.as_f64(both), ref, "bf16", "two chunks")
    H.assert_close(H.as_f64(whole), ref, "bf16", "one chunk")


def test_sequences_without_new_tokens_are_skipped(pkv):
    """A batch may hold sequences whose chunk is empty this step."""
    specs = [(40, 0), (0, 33), (100, 0), (20, 70), (5, 0)]
    wl, hv, q, qs, tables, lens = _case(8, 2, specs, seed=51)
    got, st = _run(pkv, wl, hv, q, qs, tables, lens)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens), "bf16", "empty chunks")


def test_too_long_chunk_is_flagged(pkv):
    wl, hv, q, qs, tables, lens = _case(4, 4, [(0, 300)], seed=41)
    _, st = _run(pkv, wl, hv, q, qs, tables, lens, max_query_len=100)
    assert st & 64                                   # PA_DEV_BAD_QUERY_LEN


def test_unsupported_shapes_fail_loudly(pkv):
    import torch
    q = torch.zeros(4, 6, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 2, 16, D, dtype=torch.bfloat16, device="cuda")      # group 3
    qs = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PagedKVError):
        pkv.prefill(q, kc, kc, torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                    torch.tensor([4], dtype=torch.int32, device="cuda"), qs, 4)


def test_more_items_than_ctas(pkv):
    """The kernel keeps one CTA per SM and hands out (tile, KV head, sequence)
    items from a counter: 20 sequences x 16 KV heads x up to 3 tiles is several
    items per CTA, of very different lengths, some of them empty.  Every item
    must be done exactly once, on every call (the counter restarts)."""
    import torch
    rng = np.random.default_rng(77)
    specs = [(int(rng.integers(0, 40)) * 16, int(rng.integers(1, 700))) for _ in range(20)]
    wl, hv, q, qs, tables, lens = _case(16, 16, specs, seed=78)
    ref = _oracle(wl, hv, q, qs, tables, lens)
    args = (H.host_to_device(q, torch.bfloat16), H.host_to_device(hv.key_cache, torch.bfloat16),
            H.host_to_device(hv.value_cache, torch.bfloat16), torch.from_numpy(tables).cuda(),
            torch.from_numpy(lens).cuda(), torch.from_numpy(qs).cuda(), None, wl.scale)
    ws = torch.full((int(pkv.lib().pa_prefill_workspace_bytes()),), 255, dtype=torch.uint8,
                    device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(3):
        out = torch.full_like(args[0], float("nan"))
        pkv.prefill(*args, out=out, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        H.assert_close(H.as_f64(out), ref, "bf16", f"persistent prefill, call {call}")


@pytest.mark.parametrize("name", ["prefill_llama70b_chunked", "prefill_llama7b"])
def test_full_size_workload_sampled(pkv, name):
    """The bench's prefill workloads at full size, in the bench's launch
    configuration (cache write of the chunk, then pa_prefill).  Sampled rows are
    checked one by one: query row i of sequence b sits at position p = C_b + i
    and attends to positions [0, p], which is the decode of that row's query
    over a context of p + 1 tokens."""
    import torch
    pw = W.make_prefill_workload(name)
    dev = torch.device("cuda")
    q, kc, vc, kn, vn = W.prefill_device_values(pw, dev)
    tables = torch.from_numpy(pw.block_tables).to(dev)
    lens = torch.from_numpy(pw.context_lens).to(dev)
    qs = torch.from_numpy(pw.query_start).to(dev)
    pkv.cache_write(kc, vc, kn, vn, torch.from_numpy(pw.slot_mapping).to(dev))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = pkv.prefill(q, kc, vc, tables, lens, qs, int(pw.chunk.max()), 1.0 / np.sqrt(pw.head_dim),
                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(5)
    seqs = rng.choice(pw.num_seqs, size=3, replace=False)
    rows, ctx, tabs = [], [], []
    for b in seqs:
        for i in rng.choice(int(pw.chunk[b]), size=4, replace=False):
            rows.append(int(pw.query_start[b]) + int(i))
            ctx.append(int(pw.cached[b]) + int(i) + 1)
            tabs.append(pw.block_tables[b])
    idx = torch.tensor(rows, device=dev)
    qh = H.device_to_host_bits(q.index_select(0, idx))
    kch, vch = H.device_to_host_bits(kc), H.device_to_host_bits(vc)
    ref = oracle.paged_decode(qh, kch, vch, np.stack(tabs).astype(np.int32),
                              np.asarray(ctx, np.int32), 1.0 / np.sqrt(pw.head_dim), threads=8)
    got = H.as_f64(out.index_select(0, idx))
    H.assert_close(got, ref, "bf16", f"{name} sampled rows")


def test_large_values_within_f16_range(pkv):
    """P.V runs on f16 operands: V is converted from bf16 in shared memory, exact
    for magnitudes up to 65504.  Values of a few thousand to 40000 must come
    through within the tolerance.  (They are positive: a weight's f16 rounding
    moves an output by up to 2^-11 of the largest |v| it weighs, which a
    cancelling mix of such values would not keep within 1e-2 of the result.)"""
    specs = [(0, 40), (100, 130)]
    wl, hv, q, qs, tables, lens = _case(8, 2, specs, seed=61)
    rng = np.random.default_rng(62)
    v = W.bf16_bits_to_f32(hv.value_cache)
    big = rng.choice([30000.0, 3000.0, 2500.0, 40000.0], size=v.shape).astype(np.float32)
    keep = np.isnan(v)                                  # slots outside every context stay NaN
    hv.value_cache = np.where(keep, hv.value_cache, W.to_bf16_bits(big))
    got, st = _run(pkv, wl, hv, q, qs, tables, lens)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens), "bf16", "large V")


# Key rows scaled up at some positions make those scores jump by tens of log2
# units in a later K/V tile: a 32-column chunk's weights then overflow the
# reference the row carries from the tiles before, and the chunk is computed
# again against a higher one.  [288, 320) is the second chunk of the first
# thread of the third tile (its first chunk is rescaled afterwards), [320, 384)
# the second thread's columns (the first thread's chunks follow it), [130, 140)
# a jump within the second tile.
@pytest.mark.parametrize("hq,hkv", [(8, 2), (8, 8)])
@pytest.mark.parametrize("lo,hi,factor", [(288, 320, 8.0), (320, 384, 8.0), (130, 140, 30.0),
                                          (0, 128, 8.0)])
def test_scores_rising_in_later_tiles(pkv, hq, hkv, lo, hi, factor):
    specs = [(0, 400), (200, 250), (100, 60)]
    wl, hv, q, qs, tables, lens = _case(hq, hkv, specs, seed=71 + lo)
    k = W.bf16_bits_to_f32(hv.key_cache)
    for b in range(len(specs)):
        for pos in range(lo, min(hi, int(lens[b]))):
            phys = int(tables[b, pos // 16])
            k[phys, :, pos % 16] *= np.float32(factor)
    keep = np.isnan(k)
    hv.key_cache = np.where(keep, hv.key_cache, W.to_bf16_bits(k))
    got, st = _run(pkv, wl, hv, q, qs, tables, lens)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens), "bf16",
                   f"keys x{factor} at [{lo}, {hi})")


def test_scores_rising_with_a_negative_scale(pkv):
    """The same jump seen through a negative scale: the smallest raw scores win."""
    specs = [(0, 400), (150, 200)]
    wl, hv, q, qs, tables, lens = _case(8, 2, specs, seed=91)
    k = W.bf16_bits_to_f32(hv.key_cache)
    for b in range(len(specs)):
        for pos in range(300, 340):
            phys = int(tables[b, pos // 16])
            k[phys, :, pos % 16] *= np.float32(-8.0)
    keep = np.isnan(k)
    hv.key_cache = np.where(keep, hv.key_cache, W.to_bf16_bits(k))
    got, st = _run(pkv, wl, hv, q, qs, tables, lens, scale=-0.0883883)
    assert st == 0
    H.assert_close(H.as_f64(got), _oracle(wl, hv, q, qs, tables, lens, scale=-0.0883883), "bf16",
                   "negative scale, keys x-8 at [300, 340)")
