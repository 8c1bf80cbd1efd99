"""Pins for the oracle's FP8 (E4M3) paths, against torch's float8_e4m3fn and closed forms.

The pages name FP8 KV caches ("KV cache: la memoria de trabajo que sostiene la
inferencia LLM", section "Trucos para que el cuaderno sea más fino"); the format
is E4M3 ("E4M3FN") of the OCP 8-bit floating point specification.  Quantisation
here rounds to nearest (ties to even) and saturates at +-448; torch's conversion
rounds the same way but turns values of 464 and above into NaN, so the two are
compared below 464 and the saturation is pinned by its closed form.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _torch_codes(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_every_code_value_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    # closed forms: largest finite, smallest subnormal, smallest normal, NaN codes
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])


def test_encode_matches_torch_below_overflow():
    rng = np.random.default_rng(0)
    parts = [rng.standard_normal(20000).astype(np.float32) * s for s in (1e-3, 0.05, 1, 30, 150)]
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_value(codes)
    finite = np.sort(np.unique(np.abs(vals[~np.isnan(vals)])))
    mids = ((finite[1:] + finite[:-1]) / 2).astype(np.float32)      # exact ties
    parts += [finite.astype(np.float32), mids, -mids, np.nextafter(mids, np.float32(0)),
              np.nextafter(mids, np.float32(1e9))]
    x = np.concatenate(parts)
    x = x[np.abs(x) < 464.0]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_codes(x))


def test_encode_saturates_and_keeps_nan():
    x = np.array([448, 449, 463.9, 464, 1e6, np.inf, -448, -5e4, -np.inf], np.float32)
    assert oracle.e4m3_encode(x).tolist() == [0x7E] * 6 + [0xFE] * 3
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_every_finite_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    finite = ~np.isnan(vals)
    assert np.array_equal(oracle.e4m3_encode(vals[finite]), codes[finite])


def _fp8_case(rng, B, Hq, Hkv, D, lens):
    wl = W.custom_workload(B, Hq, Hkv, D, lens, dtype="bf16", seed=int(rng.integers(1 << 30)))
    NB = wl.num_blocks
    kc = rng.integers(0, 256, size=(NB, Hkv, 16, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(NB, Hkv, 16, D), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x38        # no NaN codes in the pools
    vc[(vc & 0x7F) == 0x7F] = 0x30
    ks = rng.uniform(0.002, 0.05, Hkv).astype(np.float32)
    vs = rng.uniform(0.002, 0.05, Hkv).astype(np.float32)
    q = W.to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    return wl, q, kc, vc, ks, vs


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 4, 64), (8, 2, 128)])
def test_fp8_decode_equals_library_attention_on_dequantised_values(Hq, Hkv, D):
    rng = np.random.default_rng(Hq + D)
    lens = [1, 17, 90]
    wl, q, kc, vc, ks, vs = _fp8_case(rng, 3, Hq, Hkv, D, lens)
    got = oracle.paged_decode(q, kc, vc, wl.block_tables, wl.context_lens, 0.3,
                              k_scales=ks, v_scales=vs)
    kd = torch.from_numpy(kc).view(torch.float8_e4m3fn).double() * torch.from_numpy(
        ks.astype(np.float64))[None, :, None, None]
    vd = torch.from_numpy(vc).view(torch.float8_e4m3fn).double() * torch.from_numpy(
        vs.astype(np.float64))[None, :, None, None]
    qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).double()
    for b, L in enumerate(lens):
        rows = [(wl.block_tables[b, t // 16], t % 16) for t in range(L)]
        k = torch.stack([kd[p, :, o] for p, o in rows], dim=1)[None]      # [1,Hkv,L,D]
        v = torch.stack([vd[p, :, o] for p, o in rows], dim=1)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qd[b][None, :, None, :], k, v, scale=0.3, enable_gqa=Hq != Hkv)[0, :, 0].numpy()
        np.testing.assert_allclose(got[b], ref, rtol=1e-11, atol=1e-12)


def test_fp8_cache_write_codes_match_torch_quantisation():
    rng = np.random.default_rng(5)
    wl = W.custom_workload(4, 8, 4, 128, [3, 16, 40, 7], dtype="bf16", seed=3)
    hv = W.host_values(wl, poison_unused=False)
    kc = np.zeros((wl.num_blocks, 4, 16, 128), np.uint8)
    vc = np.zeros_like(kc)
    ks = rng.uniform(0.01, 0.03, 4).astype(np.float32)
    vs = rng.uniform(0.01, 0.03, 4).astype(np.float32)
    oracle.cache_write_fp8(kc, vc, hv.key_new, hv.value_new, wl.slot_mapping, ks, vs)
    kx = W.bf16_bits_to_f32(hv.key_new)
    vx = W.bf16_bits_to_f32(hv.value_new)
    for i, s in enumerate(wl.slot_mapping):
        qk = (kx[i] / ks[:, None]).astype(np.float32)          # IEEE float32 quotients
        qv = (vx[i] / vs[:, None]).astype(np.float32)
        assert np.all(np.abs(qk) < 464) and np.all(np.abs(qv) < 464)
        assert np.array_equal(kc[s // 16, :, s % 16], _torch_codes(qk))
        assert np.array_equal(vc[s // 16, :, s % 16], _torch_codes(qv))
    written = {(s // 16, s % 16) for s in wl.slot_mapping}
    for blk in range(wl.num_blocks):
        for off in range(16):
            if (blk, off) not in written:
                assert not kc[blk, :, off].any() and not vc[blk, :, off].any()
