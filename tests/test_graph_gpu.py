"""Library calls captured in a CUDA graph and replayed give the same bytes as the
same calls made directly.

A serving loop captures its decode step once and replays it; the bench times
replays too.  The kernels chain through programmatic dependent launches (the
shared-prefix decode lets its suffix kernel start beside the prefix kernel, and
only the suffix grid's last CTA waits for it), and a graph keeps those
dependencies as programmatic edges.  Each case runs one whole step (cache write,
copy-on-write where the workload has pairs, decode) directly, restores the
pools, captures the same calls, replays them twice, and requires the output,
both pools and the status word to match bit for bit.  The direct calls are
checked against the oracle by the other GPU tests.
"""
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_100_gb300.build import build
    build()
    import paged_kv_cache_100_gb300 as m
    return m


def _split_k_workload():
    # 8 sequences, 32 query / 8 KV heads, contexts up to 6000 tokens: several
    # 512-token partitions per sequence and the merge kernel
    lens = [6000, 1, 513, 4097, 2222, 16, 5000, 800]
    return W.custom_workload(len(lens), 32, 8, 128, lens, dtype="bf16", seed=5)


CASES = [("shared_prefix", "bf16"), ("shared_prefix", "fp8"), ("split_k", "bf16"),
         ("split_k", "fp8")]


@pytest.mark.parametrize("name,kvd", CASES)
def test_graph_replay_matches_direct_calls(pkv, name, kvd):
    import torch
    dev = torch.device("cuda", 0)
    wl = W.make_workload("shared_prefix", seed=3) if name == "shared_prefix" else _split_k_workload()
    fp8 = kvd == "fp8"
    if fp8:
        q, kc, vc, kn, vn, ks, vs = W.fp8_device_values(wl, dev, seed=9)
    else:
        q, kc, vc, kn, vn = W.device_values(wl, dev, seed=9)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    # the step writes the token at position context_lens[b] into its slot and
    # attends over context_lens[b] + 1 tokens
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    lens = torch.from_numpy(wl.step_context_lens).to(dev)
    pairs = torch.from_numpy(wl.cow_pairs).to(dev)
    n_prefix = pkv.shared_prefix_blocks(wl.block_tables) if name == "shared_prefix" else 0
    if name == "shared_prefix":
        P = wl.partition_size
        f = (pkv.lib().pa_decode_shared_prefix_fp8_workspace_bytes if fp8
             else pkv.lib().pa_decode_shared_prefix_workspace_bytes)
        need = f(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.max_blocks, n_prefix, P)
    else:
        P = 512
        need = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                          wl.max_blocks, P, kvd)
    ws = torch.empty(max(int(need), 16), dtype=torch.uint8, device=dev)
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        if fp8:
            pkv.cache_write_fp8(kc, vc, kn, vn, slots, ks, vs, status=status)
        else:
            pkv.cache_write(kc, vc, kn, vn, slots, status=status)
        if wl.cow_pairs.shape[0]:
            pkv.block_copy(kc, vc, pairs, status=status)
        if n_prefix and fp8:
            pkv.decode_shared_prefix_fp8(q, kc, vc, ks, vs, bt, lens, n_prefix, wl.scale, out=out,
                                         partition_size=P, workspace=ws, status=status)
        elif n_prefix:
            pkv.decode_shared_prefix(q, kc, vc, bt, lens, n_prefix, wl.scale, out=out,
                                     partition_size=P, workspace=ws, status=status)
        elif fp8:
            pkv.decode_fp8(q, kc, vc, ks, vs, bt, lens, wl.scale, out=out, partition_size=P,
                           workspace=ws, status=status)
        else:
            pkv.decode(q, kc, vc, bt, lens, wl.scale, out=out, partition_size=P, workspace=ws,
                       status=status)

    kc0, vc0 = kc.clone(), vc.clone()
    step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_out, want_k, want_v = out.clone(), kc.clone(), vc.clone()
    assert not torch.isnan(want_out.float()).any()

    kc.copy_(kc0)
    vc.copy_(vc0)
    out.fill_(float("nan"))
    ws.fill_(0xff)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = pkv.launch_count()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        step()
    assert pkv.launch_count() > n0          # the library's kernels were captured
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out.view(torch.int16), want_out.view(torch.int16))
        assert torch.equal(kc.view(torch.uint8), want_k.view(torch.uint8))
        assert torch.equal(vc.view(torch.uint8), want_v.view(torch.uint8))
        out.fill_(float("nan"))
