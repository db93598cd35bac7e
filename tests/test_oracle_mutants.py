"""Planted mistakes in the oracle must make its pins fail.

Each case edits one line of a copy of kv_oracle.c (a dropped term, a wrong sign, a wrong index,
a swapped operand), compiles it on the CPU, routes the oracle through that build and runs the
pins.  A mutant that no pin catches would mean the pins do not constrain that part of the
oracle.  The shipped oracle source is never modified.
"""
import math
import os

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_prefill_pins as prefill_pins
from tests import test_oracle_int4_pins as int4_pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

MUTANTS = [
    ("gqa_map_strided", "const int32_t hq = h * g + k;", "const int32_t hq = k * Hkv + h;"),
    ("spec_positions_reversed", "const int64_t p = L - ql + i;", "const int64_t p = L - 1 - i;"),
    ("window_one_short", "p - J->window + 1 > 0 ? p - J->window + 1 : 0",
     "p - J->window + 2 > 0 ? p - J->window + 2 : 0"),
    ("scale_dropped", "s[j] = J->scale * acc;", "s[j] = acc;"),
    ("lse_sign", "J->lse[tok * Hq + hq] = m + log(den);", "J->lse[tok * Hq + hq] = m - log(den);"),
    ("v_read_from_k", "V[j * D + d] = elem_to_double(J->v_cache", "V[j * D + d] = elem_to_double(J->k_cache"),
    ("gather_offset", "(physical * bs + j % bs) * Hkv + h", "(physical * bs + (j + 1) % bs) * Hkv + h"),
    ("gather_block_index", "J->block_table[(int64_t)b * J->bt_stride + j / bs]",
     "J->block_table[(int64_t)b * J->bt_stride + j / bs / 2]"),
    ("slot_offset", "slot_mapping[t] = physical * block_size + offset;",
     "slot_mapping[t] = physical * block_size + logical;"),
    ("slot_row", "block_table[(int64_t)r * bt_stride + logical]",
     "block_table[(int64_t)(r > 0 ? r - 1 : 0) * bt_stride + logical]"),
    ("write_offset", "offset = slot % block_size;", "offset = (slot + 1) % block_size;"),
    ("e4m3_bias", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3_subnormal_scale", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("e4m3_truncates", "double q = nearbyint(ldexp(a, 3 - e));", "double q = floor(ldexp(a, 3 - e));"),
    ("e4m3_no_saturation", "if (a >= 448.0)\n        return (uint8_t)(sign | 0x7e);",
     "if (a >= 464.0)\n        return (uint8_t)(sign | 0x7f);"),
    ("bf16_exponent", "v = ldexp(1.0 + m / 128.0, e - 127);", "v = ldexp(1.0 + m / 128.0, e - 126);"),
    ("f16_mantissa", "v = ldexp(1.0 + m / 1024.0, e - 15);", "v = ldexp(1.0 + m / 512.0, e - 15);"),
    ("fp8_write_scale", "orc_e4m3_from_float(kx / k_scale)", "orc_e4m3_from_float(kx * k_scale)"),
    ("varlen_row_offset", "J->query_start_loc ? J->query_start_loc[b] : (int64_t)b * J->q_len",
     "J->query_start_loc ? (int64_t)b * (J->query_start_loc[b + 1] - J->query_start_loc[b]) : (int64_t)b * J->q_len"),
    ("varlen_count", "J->query_start_loc[b + 1] - row0 : J->q_len",
     "J->query_start_loc[b + 1] - row0 - (b > 0) : J->q_len"),
    ("window_first_key_read", "J->window > 0 && L - ql - J->window + 1 > 0 ? L - ql - J->window + 1 : 0",
     "J->window > 0 && L - J->window + 1 > 0 ? L - J->window + 1 : 0"),
    ("int4_nibble_order", "return (idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);",
     "return (idx & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);"),
    ("int4_put_order", "if (idx & 1)\n        *byte = (uint8_t)((*byte & 0x0F) | (nibble << 4));",
     "if (!(idx & 1))\n        *byte = (uint8_t)((*byte & 0x0F) | (nibble << 4));"),
    ("int4_truncates", "double q = nearbyint((double)x);", "double q = trunc((double)x);"),
    ("int4_no_saturation", "if (q > 7.0)\n        q = 7.0;", "if (q > 8.0)\n        q = 8.0;"),
    ("int4_sign", "return (double)(n >= 8 ? n - 16 : n);", "return (double)(n >= 8 ? n - 8 : n);"),
    ("int4_write_scale", "orc_int4_from_float(kx / ks)", "orc_int4_from_float(kx * ks)"),
    ("int4_write_group", "float vs = v_scales[h * groups + d / group_size];",
     "float vs = v_scales[h * groups + d % groups];"),
    ("int4_read_group", "ksc = J->k_gscales[(int64_t)h * (D / J->group_size) + d / J->group_size];",
     "ksc = J->k_gscales[(int64_t)h * (D / J->group_size) + d % (D / J->group_size)];"),
    ("int4_v_scale_from_k", "vsc = J->v_gscales[", "vsc = J->k_gscales["),
]


def _pin_probes():
    g = GOLDEN
    yield lambda: pins.test_slot_token7_block37(g)
    yield lambda: pins.test_slot_48_tokens_three_blocks(g)
    yield lambda: pins.test_slot_worker_rows(g)
    yield lambda: pins.test_slot_block_of_4_spill(g)
    yield lambda: pins.test_slot_bruteforce_enumeration(16)
    yield lambda: pins.test_e4m3_fixed_points(g)
    yield pins.test_e4m3_decode_all_codes_vs_torch
    yield pins.test_e4m3_encode_roundtrip_and_ties
    yield pins.test_e4m3_saturation
    yield lambda: pins.test_cache_write_roundtrip_16bit("f16")
    yield lambda: pins.test_cache_write_roundtrip_16bit("bf16")
    yield pins.test_cache_write_fp8_matches_torch_conversion
    yield lambda: pins.test_attention_matches_sdpa("f16", 4, 2, 16, 4, 1, 0)
    yield lambda: pins.test_attention_matches_sdpa("bf16", 8, 2, 32, 8, 3, 0)
    yield lambda: pins.test_attention_matches_sdpa("bf16", 8, 1, 16, 4, 4, 5)
    yield pins.test_attention_closed_forms
    yield pins.test_attention_fp8_cache_matches_sdpa_on_dequantised_cache
    yield lambda: prefill_pins.test_prefill_matches_sdpa("f16", 4, 1, 16, 4, 0)
    yield lambda: prefill_pins.test_prefill_matches_sdpa("bf16", 6, 2, 16, 4, 20)
    yield pins.test_attention_window_released_entries_are_not_read
    yield int4_pins.test_int4_decodes_all_16_codes
    yield int4_pins.test_int4_encode_rounds_half_to_even_and_saturates
    yield lambda: int4_pins.test_int4_cache_write_matches_numpy_quantisation(32)
    yield lambda: int4_pins.test_int4_attention_matches_sdpa_on_dequantised_cache(8, 2, 1, 0, 32)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} must match exactly once"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    caught = []
    with oracle.using_library(lib):
        for probe in _pin_probes():
            try:
                probe()
            except (AssertionError, ValueError):
                caught.append(probe)
                break
    assert caught, f"planted mistake '{name}' passed every pin"
