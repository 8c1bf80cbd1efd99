"""Seeded synthetic inputs for paged decode attention.

This module only draws inputs: sequence lengths, block tables built from a
shuffled pool, slot lists and normally distributed Q/K/V values.  It holds none
of the attention, cache-write or block-copy arithmetic, so the oracle and the
CUDA path can both be fed from it without sharing any of that code.

Workloads (all block_size 16, layout [num_blocks][num_kv_heads][16][head_dim]):

  tiny           1 layer, 4 heads MHA, head_dim 64, fp32, 4 sequences with
                 context lengths {1, 17, 33, 64}, a 16-block pool assigned by a
                 seeded permutation, values N(0, 1), scale 1/8.
  llama7b_mha    32 heads MHA, head_dim 128, bf16, batch 64, context lengths
                 uniform in [128, 2048], pool 1.1x the blocks in use, block
                 tables are contiguous slices of a shuffled pool, values N(0, 1).
  llama70b_gqa   64 query / 8 KV heads, head_dim 128, bf16, batch 256, context
                 lengths uniform in [512, 4096], values N(0, 0.5) (0.5 read as
                 the standard deviation).
  long_splitk    32 heads MHA, head_dim 128, bf16, batch 8, context 32768 for
                 every sequence, split-K partitions of 512 tokens, values N(0, 1).
  shared_prefix  32 query / 8 KV heads, head_dim 128, bf16, batch 128; every
                 block table starts with the same 64 blocks (a 1024-token
                 prefix) followed by its own suffix blocks (suffix lengths
                 uniform in [16, 1024]); the first 16 sequences get a private
                 copy of the last prefix block (copy-on-write pairs).

A decode step appends one new token per sequence at position ``context_lens[b]``
(its slot is in ``slot_mapping``) and then attends over ``context_lens[b] + 1``
tokens.  The tables therefore already hold the block that position needs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f32" or "bf16"
    value_std: float
    context_lens: np.ndarray        # int32 [B]: tokens already in the cache
    block_tables: np.ndarray        # int32 [B][max_blocks]; -1 past the used entries
    num_blocks: int
    slot_mapping: np.ndarray        # int64 [B]: slot of the appended token
    cow_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int32))
    partition_size: int = 0         # 0 = the library's choice
    seed: int = 0
    block_size: int = BLOCK_SIZE

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]

    @property
    def step_context_lens(self) -> np.ndarray:
        """Context lengths seen by the decode that follows the step's append."""
        return (self.context_lens + 1).astype(np.int32)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def pool_shape(self):
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)


def _blocks(n_tokens) -> np.ndarray:
    return -(-np.asarray(n_tokens, dtype=np.int64) // BLOCK_SIZE)


def _tables_from_slices(order: np.ndarray, need: np.ndarray) -> np.ndarray:
    """Block tables made of consecutive slices of ``order`` (one slice per sequence)."""
    B = need.shape[0]
    width = int(need.max()) if B else 0
    tables = np.full((B, width), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        n = int(need[b])
        tables[b, :n] = order[pos:pos + n]
        pos += n
    return tables


def _append_slots(tables: np.ndarray, lens: np.ndarray) -> np.ndarray:
    B = lens.shape[0]
    pos = lens.astype(np.int64)
    phys = tables[np.arange(B), pos // BLOCK_SIZE].astype(np.int64)
    return phys * BLOCK_SIZE + pos % BLOCK_SIZE


def make_workload(name: str, seed: int = 0) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "tiny":
        lens = np.array([1, 17, 33, 64], dtype=np.int32)
        num_blocks = 16
        order = rng.permutation(num_blocks).astype(np.int32)
        need = _blocks(lens + 1)          # room for the appended token too
        tables = _tables_from_slices(order, need)
        return Workload(name, 4, 4, 4, 64, "f32", 1.0, lens, tables, num_blocks,
                        _append_slots(tables, lens), seed=seed)

    if name in ("llama7b_mha", "llama70b_gqa", "long_splitk"):
        if name == "llama7b_mha":
            B, Hq, Hkv, std = 64, 32, 32, 1.0
            lens = rng.integers(128, 2048, size=B, endpoint=True).astype(np.int32)
        elif name == "llama70b_gqa":
            B, Hq, Hkv, std = 256, 64, 8, 0.5
            lens = rng.integers(512, 4096, size=B, endpoint=True).astype(np.int32)
        else:
            B, Hq, Hkv, std = 8, 32, 32, 1.0
            lens = np.full(B, 32768, dtype=np.int32)
        need = _blocks(lens + 1)
        num_blocks = int(math.ceil(1.1 * int(need.sum())))
        order = rng.permutation(num_blocks).astype(np.int32)
        tables = _tables_from_slices(order, need)
        return Workload(name, B, Hq, Hkv, 128, "bf16", std, lens, tables, num_blocks,
                        _append_slots(tables, lens),
                        partition_size=512 if name == "long_splitk" else 0, seed=seed)

    if name == "shared_prefix":
        B, Hq, Hkv, prefix_blocks, n_cow = 128, 32, 8, 64, 16
        suffix = rng.integers(16, 1024, size=B, endpoint=True).astype(np.int64)
        lens = (prefix_blocks * BLOCK_SIZE + suffix).astype(np.int32)
        own = _blocks(lens.astype(np.int64) + 1) - prefix_blocks
        used = prefix_blocks + int(own.sum()) + n_cow
        num_blocks = int(math.ceil(1.1 * used))
        order = rng.permutation(num_blocks).astype(np.int32)
        prefix = order[:prefix_blocks]
        suffix_tables = _tables_from_slices(order[prefix_blocks:], own)
        width = prefix_blocks + suffix_tables.shape[1]
        tables = np.full((B, width), -1, dtype=np.int32)
        tables[:, :prefix_blocks] = prefix
        tables[:, prefix_blocks:] = suffix_tables
        fresh = order[prefix_blocks + int(own.sum()):prefix_blocks + int(own.sum()) + n_cow]
        cow = np.stack([np.full(n_cow, prefix[-1], dtype=np.int32), fresh], axis=1)
        tables[:n_cow, prefix_blocks - 1] = fresh   # these sequences read their copy
        return Workload(name, B, Hq, Hkv, 128, "bf16", 1.0, lens, tables, num_blocks,
                        _append_slots(tables, lens), cow_pairs=cow.astype(np.int32), seed=seed)

    raise KeyError(f"unknown workload {name!r}")


WORKLOADS = ("tiny", "llama7b_mha", "llama70b_gqa", "long_splitk", "shared_prefix")


# ---------------------------------------------------------------------------
# Chunked prefill ("PagedAttention por dentro", section "Chunked prefill
# integrado con paged KV")
# ---------------------------------------------------------------------------
@dataclass
class PrefillWorkload:
    """Sequences that each bring a chunk of new tokens on top of a cached context."""
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    value_std: float
    cached: np.ndarray              # int32 [B]: tokens already in the cache
    chunk: np.ndarray               # int32 [B]: new tokens of this step
    block_tables: np.ndarray        # int32 [B][max_blocks]
    num_blocks: int
    seed: int = 0
    dtype: str = "bf16"
    block_size: int = BLOCK_SIZE

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]

    @property
    def elem_bytes(self) -> int:
        return 2

    @property
    def context_lens(self) -> np.ndarray:
        return (self.cached + self.chunk).astype(np.int32)

    @property
    def query_start(self) -> np.ndarray:
        qs = np.zeros(self.num_seqs + 1, dtype=np.int32)
        qs[1:] = np.cumsum(self.chunk)
        return qs

    @property
    def num_tokens(self) -> int:
        return int(self.chunk.sum())

    @property
    def slot_mapping(self) -> np.ndarray:
        """int64 [num_tokens]: slot of every chunk token (positions C .. C+T-1)."""
        out = []
        for b in range(self.num_seqs):
            pos = np.arange(int(self.cached[b]), int(self.cached[b] + self.chunk[b]), dtype=np.int64)
            out.append(self.block_tables[b, pos // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE
                       + pos % BLOCK_SIZE)
        return np.concatenate(out) if out else np.zeros(0, np.int64)

    def pool_shape(self):
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)


def make_prefill_workload(name: str, seed: int = 0) -> PrefillWorkload:
    """prefill_llama7b: 8 fresh 2048-token prompts, 32 heads MHA, head_dim 128;
    prefill_llama70b_chunked: 16 sequences of 64 query / 8 KV heads, each bringing a
    512-token chunk on top of a cached context uniform in [0, 8192] (multiples of
    16).  bf16, N(0, 1) values, tables are slices of a shuffled pool 1.1x the blocks
    in use."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "prefill_llama7b":
        B, Hq, Hkv, std = 8, 32, 32, 1.0
        cached = np.zeros(B, dtype=np.int32)
        chunk = np.full(B, 2048, dtype=np.int32)
    elif name == "prefill_llama70b_chunked":
        B, Hq, Hkv, std = 16, 64, 8, 1.0
        cached = (rng.integers(0, 512, size=B, endpoint=True) * 16).astype(np.int32)
        chunk = np.full(B, 512, dtype=np.int32)
    elif name == "prefill_tiny":
        B, Hq, Hkv, std = 3, 8, 2, 1.0
        cached = np.array([0, 37, 200], dtype=np.int32)
        chunk = np.array([70, 19, 130], dtype=np.int32)
    else:
        raise KeyError(f"unknown prefill workload {name!r}")
    need = _blocks(cached.astype(np.int64) + chunk)
    num_blocks = int(math.ceil(1.1 * int(need.sum()))) + 1
    order = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_slices(order, need)
    return PrefillWorkload(name, B, Hq, Hkv, 128, std, cached, chunk, tables, num_blocks, seed)


PREFILL_WORKLOADS = ("prefill_llama7b", "prefill_llama70b_chunked", "prefill_tiny")


def prefill_device_values(pw: PrefillWorkload, device, seed: int | None = None):
    """(query, key_cache, value_cache, key_new, value_new) in bf16 on a CUDA device,
    drawn with a seeded torch generator (values N(0, value_std))."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(pw.seed + 7 if seed is None else seed)

    def draw(shape):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        return (x * pw.value_std).to(torch.bfloat16)

    N = pw.num_tokens
    q = draw((N, pw.num_q_heads, pw.head_dim))
    kc = draw(pw.pool_shape())
    vc = draw(pw.pool_shape())
    kn = draw((N, pw.num_kv_heads, pw.head_dim))
    vn = draw((N, pw.num_kv_heads, pw.head_dim))
    return q, kc, vc, kn, vn


def custom_workload(num_seqs, num_q_heads, num_kv_heads, head_dim, context_lens, dtype="bf16",
                    value_std=1.0, spare_blocks=4, seed=0, name="custom") -> Workload:
    """A workload with given lengths; block tables are slices of a shuffled pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(context_lens, dtype=np.int32).reshape(num_seqs)
    need = _blocks(lens.astype(np.int64) + 1)
    num_blocks = int(need.sum()) + int(spare_blocks)
    order = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_slices(order, need)
    return Workload(name, num_seqs, num_q_heads, num_kv_heads, head_dim, dtype, value_std, lens,
                    tables, num_blocks, _append_slots(tables, lens), seed=seed)


# ---------------------------------------------------------------------------
# Values
# ---------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); returns uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class HostValues:
    query: np.ndarray        # [B][Hq][D]   float32 or uint16 (bf16 bits)
    key_cache: np.ndarray    # [NB][Hkv][16][D]
    value_cache: np.ndarray
    key_new: np.ndarray      # [B][Hkv][D]  the appended token's K
    value_new: np.ndarray


def host_values(wl: Workload, seed: int | None = None, poison_unused: bool = True) -> HostValues:
    """Normally distributed values drawn on the host (numpy PCG64).

    With ``poison_unused`` every slot that holds no context token (past the last
    token of each sequence, and blocks no table uses) is filled with NaN, so a
    kernel that reads one shows it in its output.
    """
    rng = np.random.Generator(np.random.PCG64(wl.seed + 1 if seed is None else seed))
    B, Hq, Hkv, D = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim

    def draw(shape):
        return (rng.standard_normal(shape, dtype=np.float32) * np.float32(wl.value_std))

    q = draw((B, Hq, D))
    kc = draw(wl.pool_shape())
    vc = draw(wl.pool_shape())
    kn = draw((B, Hkv, D))
    vn = draw((B, Hkv, D))
    if poison_unused:
        mask = used_slot_mask(wl)
        kc[~mask] = np.nan
        vc[~mask] = np.nan
    if wl.dtype == "bf16":
        q, kc, vc, kn, vn = (to_bf16_bits(a) for a in (q, kc, vc, kn, vn))
    return HostValues(q, kc, vc, kn, vn)


def used_slot_mask(wl: Workload, lens=None) -> np.ndarray:
    """bool [NB][16]: True where a slot holds one of the first ``lens[b]`` tokens."""
    lens = wl.context_lens if lens is None else np.asarray(lens)
    mask = np.zeros((wl.num_blocks, wl.block_size), dtype=bool)
    for b in range(wl.num_seqs):
        L = int(lens[b])
        nb = -(-L // wl.block_size)
        for j in range(nb):
            phys = int(wl.block_tables[b, j])
            fill = min(wl.block_size, L - j * wl.block_size)
            mask[phys, :fill] = True
    return mask[:, None, :].repeat(wl.num_kv_heads, axis=1)


def device_values(wl: Workload, device, seed: int | None = None):
    """The same kinds of values drawn on a CUDA device with a seeded torch generator.

    Returns torch tensors (query, key_cache, value_cache, key_new, value_new) in the
    workload's dtype.  Used where the pools are too large to draw on the host.
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed + 1 if seed is None else seed)
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    B, Hq, Hkv, D = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim

    def draw(shape):
        out = torch.empty(shape, dtype=tdt, device=device)
        flat = out.view(-1)
        chunk = 1 << 26
        for s in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - s)
            tmp = torch.randn(n, generator=g, device=device, dtype=torch.float32)
            flat[s:s + n].copy_(tmp.mul_(wl.value_std))
        return out

    return (draw((B, Hq, D)), draw(wl.pool_shape()), draw(wl.pool_shape()),
            draw((B, Hkv, D)), draw((B, Hkv, D)))


# ---------------------------------------------------------------------------
# FP8 (E4M3) pools
# ---------------------------------------------------------------------------
FP8_RANGE_SIGMAS = 8.0      # +-8 standard deviations map to the largest code, 448


def fp8_scales(wl: Workload) -> np.ndarray:
    """Per-KV-head scales: a stored code stands for code_value * scale."""
    return np.full(wl.num_kv_heads, FP8_RANGE_SIGMAS * wl.value_std / 448.0, dtype=np.float32)


def to_e4m3_codes(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """E4M3 codes of x / scale (per KV head on axis 1), clamped to +-448 first."""
    import torch
    s = np.asarray(scale, np.float32).reshape((1, -1) + (1,) * (x.ndim - 2))
    q = np.clip(np.asarray(x, np.float32) / s, -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@dataclass
class Fp8HostValues:
    query: np.ndarray        # [B][Hq][D] bf16 bits
    key_cache: np.ndarray    # [NB][Hkv][16][D] E4M3 codes
    value_cache: np.ndarray
    key_new: np.ndarray      # [B][Hkv][D] bf16 bits (quantised by the cache write)
    value_new: np.ndarray
    k_scales: np.ndarray     # [Hkv] float32
    v_scales: np.ndarray


def fp8_host_values(wl: Workload, seed: int | None = None, poison_unused: bool = True):
    """Host values for FP8 pools: normal values quantised to E4M3 per KV head; with
    ``poison_unused`` the slots holding no context token get the NaN code 0x7F."""
    hv = host_values(wl, seed=seed, poison_unused=False)
    f = bf16_bits_to_f32 if hv.key_cache.dtype == np.uint16 else (lambda a: a)
    ks = fp8_scales(wl)
    vs = fp8_scales(wl)
    kc = to_e4m3_codes(f(hv.key_cache), ks)
    vc = to_e4m3_codes(f(hv.value_cache), vs)
    if poison_unused:
        mask = used_slot_mask(wl)
        kc[~mask] = 0x7F
        vc[~mask] = 0x7F
    q, kn, vn = hv.query, hv.key_new, hv.value_new
    if q.dtype != np.uint16:
        q, kn, vn = to_bf16_bits(q), to_bf16_bits(kn), to_bf16_bits(vn)
    return Fp8HostValues(q, kc, vc, kn, vn, ks, vs)


def fp8_device_values(wl: Workload, device, seed: int | None = None):
    """(query bf16, key_cache uint8, value_cache uint8, key_new bf16, value_new bf16,
    k_scales, v_scales) drawn on a CUDA device with a seeded torch generator."""
    import torch
    q, kc, vc, kn, vn = device_values(wl, device, seed=seed)
    ks = torch.from_numpy(fp8_scales(wl)).to(device)
    vs = torch.from_numpy(fp8_scales(wl)).to(device)

    def quant(pool, s):
        out = torch.empty(pool.shape, dtype=torch.uint8, device=device)
        for b0 in range(0, pool.shape[0], 4096):
            x = pool[b0:b0 + 4096].float() / s.view(1, -1, 1, 1)
            out[b0:b0 + 4096] = x.clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        return out

    return q, quant(kc, ks), quant(vc, vs), kn, vn, ks, vs
