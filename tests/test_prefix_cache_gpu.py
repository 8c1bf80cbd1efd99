"""Prefix caching end to end on the GPU: a request that reuses cached blocks decodes
exactly like one that wrote every position itself."""
import numpy as np
import pytest

import oracle
from tests import helpers as H

pytestmark = pytest.mark.gpu

HKV, HQ, D = 4, 16, 128


def _rows(tokens, positions):
    """K/V rows that depend only on (token id, position), as a model's would."""
    k = np.empty((len(tokens), HKV, D), np.float32)
    v = np.empty_like(k)
    for i, (tok, pos) in enumerate(zip(tokens, positions)):
        rng = np.random.default_rng(int(tok) * 100003 + int(pos))
        k[i] = rng.standard_normal((HKV, D))
        v[i] = rng.standard_normal((HKV, D))
    from workloads import to_bf16_bits
    return to_bf16_bits(k), to_bf16_bits(v)


def _write(pkv, bm, seq, tokens, kc, vc, start):
    import torch
    table = bm.table(seq)
    pos = np.arange(start, len(tokens))
    slots = np.array([table[p // 16] * 16 + p % 16 for p in pos], np.int64)
    k, v = _rows(tokens[start:], pos)
    pkv.cache_write(kc, vc, H.host_to_device(k, torch.bfloat16), H.host_to_device(v, torch.bfloat16),
                    torch.from_numpy(slots).cuda())


def _decode(pkv, bm, seq, L, q, kc, vc):
    import torch
    t = np.array([bm.table(seq)], np.int32)
    out = pkv.decode(q, kc, vc, torch.from_numpy(t).cuda(),
                     torch.tensor([L], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    return out, t


def test_reused_prefix_blocks_decode_identically():
    import torch
    from paged_kv_cache_100_gb300.build import build
    build()
    import paged_kv_cache_100_gb300 as pkv
    NB = 40
    rng = np.random.default_rng(0)
    tokens_a = rng.integers(0, 1000, 90).tolist()
    tokens_b = tokens_a[:70] + rng.integers(0, 1000, 25).tolist()     # 95 tokens
    q = torch.randn(1, HQ, D, dtype=torch.float32, generator=torch.Generator().manual_seed(3))
    q = q.to(torch.bfloat16).cuda()

    # cached path: A runs, is indexed and released; B reuses A's first 4 blocks
    bm = pkv.BlockManager(NB)
    kc = torch.zeros(NB, HKV, 16, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    assert bm.alloc_seq_cached(0, tokens_a) == 0
    _write(pkv, bm, 0, tokens_a, kc, vc, 0)
    assert bm.register_prefix(0, tokens_a) == 5
    table_a = bm.table(0)
    bm.free_seq(0)
    cached = bm.alloc_seq_cached(1, tokens_b)
    assert cached == 64 and bm.table(1)[:4] == table_a[:4]
    _write(pkv, bm, 1, tokens_b, kc, vc, cached)                       # only the new positions
    out_cached, t_cached = _decode(pkv, bm, 1, len(tokens_b), q, kc, vc)

    # fresh path: B alone writes every position
    bm2 = pkv.BlockManager(NB)
    kc2 = torch.zeros_like(kc)
    vc2 = torch.zeros_like(kc)
    bm2.alloc_seq(1, len(tokens_b))
    _write(pkv, bm2, 1, tokens_b, kc2, vc2, 0)
    out_fresh, _ = _decode(pkv, bm2, 1, len(tokens_b), q, kc2, vc2)

    assert torch.equal(out_cached.view(torch.int16), out_fresh.view(torch.int16))
    ref = oracle.paged_decode(H.device_to_host_bits(q), H.device_to_host_bits(kc),
                              H.device_to_host_bits(vc), t_cached,
                              np.array([len(tokens_b)], np.int32), 1 / np.sqrt(D))
    H.assert_close(H.as_f64(out_cached), ref, "bf16", "prefix-cached decode")
