"""Plant plausible mistakes in the oracle's C source and check that a pin catches each.

Each mutant is compiled from a text-edited copy of ``oracle/pa_oracle.c`` into a
temporary library, swapped in for the real one, and the pin tests of
``test_oracle_pins`` are run against it: at least one must fail.  This runs on
the CPU only.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTANTS = {
    "drop_scale": ("score[t] = scale * dot;", "score[t] = dot;"),
    "kv_head_modulo": ("v_scales, block_tables, b, h / group, first, L,",
                       "v_scales, block_tables, b, h % num_kv_heads, first, L,"),
    "prefill_excludes_self": ("h / group, first, p + 1, num_kv_heads",
                              "h / group, first, p, num_kv_heads"),
    "prefill_ignores_cached_context": ("const int p = L - T + (int)(tok - query_start[sb]);",
                                       "const int p = (int)(tok - query_start[sb]);"),
    "prefill_window_off_by_one": ("(window > 0 && p + 1 > window) ? p + 1 - window : 0;",
                                  "(window > 0 && p + 1 > window) ? p - window : 0;"),
    "prefill_kv_head": ("h / group, first, p + 1, num_kv_heads",
                        "h % num_kv_heads, first, p + 1, num_kv_heads"),
    "offset_shift": ("int offset = t % block_size;", "int offset = (t + 1) % block_size;"),
    "block_index": ("int logical_block = t / block_size;",
                    "int logical_block = (t / block_size) % 2;"),
    "short_context": ("const int L = context_lens[b];",
                      "const int L = context_lens[b] - (context_lens[b] > 1);"),
    "softmax_sign": ("double w = exp(score[t] - mx) / denom;",
                     "double w = exp(mx - score[t]) / denom;"),
    "no_normalise": ("double w = exp(score[t] - mx) / denom;", "double w = exp(score[t] - mx);"),
    "bf16_shift": ("<< 16;", "<< 15;"),
    "write_offset": ("int64_t off = s % block_size;", "int64_t off = (s + 1) % block_size;"),
    "write_skips_v": ("memcpy((char *)value_cache + dst, (const char *)value + src, (size_t)row_bytes);",
                      ";"),
    "e4m3_subnormal_step": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -8);"),
    "e4m3_bias": ("v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    "e4m3_ties_away": ("return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;", "return fl + 1.0;"),
    "e4m3_no_saturation": ("mag = 0x7E;", "mag = 0x7F;"),
    "fp8_k_scale_ignored": ("const double ks = k_scales ? (double)k_scales[kvh] : 1.0;",
                            "const double ks = 1.0;"),
    "fp8_write_multiplies": ("float kq = kx / k_scales[kvh];", "float kq = kx * k_scales[kvh];"),
    "window_off_by_one": ("const int first = (window > 0 && L > window) ? L - window : 0;",
                          "const int first = (window > 0 && L > window) ? L - window + 1 : 0;"),
    "copy_skips_v": ("memcpy((char *)value_cache + dst * block_bytes,", "(void)(value_cache + dst * block_bytes,"),
    "copy_ignores_clashes": ("        if (clash) {\n            *skipped = 1;", "        if (0) {\n            *skipped = 1;"),
    "copy_checks_dst_only": ("(pairs[2 * q] == dst || pairs[2 * q + 1] == dst)", "(pairs[2 * q + 1] == dst)"),
    "copy_self_pair_live": ("live[p] = src != dst;", "live[p] = 1;"),
}

from tests import test_oracle_fp8_pins as fp8pins  # noqa: E402

PIN_FUNCS = [
    lambda g: pins.test_prefill_matches_library_causal_attention(2, 8, 2, 64, [(0, 21), (37, 19), (100, 1)]),
    lambda g: pins.test_prefill_window_matches_library_attention(9),
    lambda g: pins.test_window_matches_library_attention_on_the_last_tokens(17),
    lambda g: fp8pins.test_every_code_value_matches_torch(),
    lambda g: fp8pins.test_encode_matches_torch_below_overflow(),
    lambda g: fp8pins.test_encode_saturates_and_keeps_nan(),
    lambda g: fp8pins.test_every_finite_code_round_trips(),
    lambda g: fp8pins.test_fp8_decode_equals_library_attention_on_dequantised_values(8, 2, 128),
    lambda g: fp8pins.test_fp8_cache_write_codes_match_torch_quantisation(),
    lambda g: pins.test_matches_library_attention_on_contiguous_tokens(4, 4, 4, 64, [1, 17, 33, 64], 0.125),
    lambda g: pins.test_matches_library_attention_on_contiguous_tokens(3, 8, 2, 128, [15, 16, 100], 0.0883883),
    lambda g: pins.test_bf16_inputs_widen_exactly(),
    lambda g: pins.test_one_token_context_returns_its_value_exactly(),
    lambda g: pins.test_zero_query_averages_the_context(),
    lambda g: pins.test_dominant_key_selects_its_token(17),
    lambda g: pins.test_worked_block_table_reads_only_its_session(g),
    lambda g: pins.test_gqa_equals_mha_with_repeated_kv_heads(),
    lambda g: pins.test_cache_write_places_each_row_in_its_slot_and_nothing_else(),
    lambda g: pins.test_cache_write_then_decode_sees_the_new_token(),
    lambda g: pins.test_block_copy_duplicates_whole_blocks_and_cow_is_invisible_to_decode(),
    lambda g: pins.test_block_copy_chained_list_skips_the_pair_that_overwrites_a_source(),
    lambda g: pins.test_block_copy_duplicate_destination_skips_both_pairs(),
    lambda g: pins.test_block_copy_self_pair_is_a_no_op_that_blocks_nothing(),
]


def _compile(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(src), "-o",
                    str(so), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, golden_dir, monkeypatch):
    text = open(SRC).read()
    old, new = MUTANTS[name]
    assert old in text, f"mutation anchor for {name} not found"
    so = _compile(tmp_path, name, text.replace(old, new))
    real = oracle._load()
    mutant = ctypes.CDLL(so)
    for fn in ("pao_paged_decode", "pao_paged_decode_ex", "pao_cache_write",
               "pao_cache_write_fp8", "pao_e4m3_value", "pao_e4m3_encode", "pao_block_copy",
               "pao_max_threads", "pao_paged_prefill"):
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
        getattr(mutant, fn).restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", mutant)
    failures = 0
    for pin in PIN_FUNCS:
        try:
            pin(golden_dir)
        except (AssertionError, ValueError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name!r}"


def test_unmutated_source_passes_every_pin(golden_dir):
    for pin in PIN_FUNCS:
        pin(golden_dir)
