"""Shared test helpers: moving seeded inputs to the device and comparing with the oracle."""
from __future__ import annotations

import numpy as np

import workloads as W

BF16_ATOL, BF16_RTOL = 2e-3, 1e-2
F32_ATOL, F32_RTOL = 1e-5, 1e-5


def torch_dtype(wl):
    import torch
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def host_to_device(arr: np.ndarray, dtype, device="cuda"):
    """float32 arrays as float32, uint16 arrays as bfloat16 bit patterns."""
    import torch
    if arr.dtype == np.uint16:
        t = torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    assert t.dtype == dtype
    return t.to(device)


def device_to_host_bits(t) -> np.ndarray:
    """A device tensor back to the oracle's representation (float32 or uint16 bits)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def as_f64(t) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def tolerance(dtype_str):
    return (F32_ATOL, F32_RTOL) if dtype_str == "f32" else (BF16_ATOL, BF16_RTOL)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype_str: str, what: str = "") -> dict:
    """Per-element |got - ref| <= atol + rtol * |ref|; returns the error summary."""
    atol, rtol = tolerance(dtype_str)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)            # NaN counts as bad
    summary = {"max_abs": float(np.nanmax(err)) if err.size else 0.0,
               "max_rel": float(np.nanmax(err / np.maximum(np.abs(ref), 1e-30))) if err.size else 0.0,
               "n_bad": int(bad.sum())}
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {summary}; first bad {idx.tolist()} got "
                             f"{got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
    return summary


def compact_for_sequences(wl, seqs, key_cache, value_cache, lens):
    """Host copies of just the blocks the given sequences read, with remapped tables.

    Returns (kc_host, vc_host, tables, lens) in the oracle's representation.
    """
    import torch
    seqs = np.asarray(seqs)
    lens = np.asarray(lens)[seqs].astype(np.int32)
    need = -(-lens.astype(np.int64) // 16)
    width = max(int(need.max()), 1)
    tabs = np.full((len(seqs), width), -1, dtype=np.int32)
    for i, b in enumerate(seqs):
        tabs[i, :need[i]] = wl.block_tables[b, :need[i]]
    used = np.unique(tabs[tabs >= 0])
    remap = np.full(wl.num_blocks, -1, dtype=np.int64)
    remap[used] = np.arange(used.size)
    new_tabs = np.where(tabs >= 0, remap[np.maximum(tabs, 0)], -1).astype(np.int32)
    idx = torch.from_numpy(used.astype(np.int64)).to(key_cache.device)
    kc = device_to_host_bits(key_cache.index_select(0, idx))
    vc = device_to_host_bits(value_cache.index_select(0, idx))
    return kc, vc, new_tabs, lens


def sample_pairs(wl, lens, n_seqs=6, heads_per_seq=4, seed=0):
    """Sequences to check (longest, shortest and random ones) and (row, head) pairs."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens)
    picks = {int(np.argmax(lens)), int(np.argmin(lens))}
    while len(picks) < min(n_seqs, wl.num_seqs):
        picks.add(int(rng.integers(wl.num_seqs)))
    seqs = sorted(picks)
    pairs = []
    for i, _ in enumerate(seqs):
        hs = {0, wl.num_q_heads - 1}
        while len(hs) < min(heads_per_seq, wl.num_q_heads):
            hs.add(int(rng.integers(wl.num_q_heads)))
        pairs += [(i, h) for h in sorted(hs)]
    return seqs, np.asarray(pairs, dtype=np.int32)
