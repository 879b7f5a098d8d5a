"""The pins must catch plausible mistakes in the oracle.

Each case copies oracle/pa_oracle.c, plants one mistake (a dropped term, a
wrong sign or index, an off-by-one, a swapped operand), compiles the copy
with gcc into a temporary library, and runs the pin that should notice it.
The planted copy never leaves the temporary directory and is CPU-only.
"""
import os

import pytest

import oracle as oracle_pkg
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "pa_oracle.c")

# (name, original snippet, planted snippet, pins expected to fail)
MUTATIONS = [
    ("offset_uses_division", "int64_t offset = position % block_size;",
     "int64_t offset = position / block_size;", ["slot_examples"]),
    ("slot_subtracts_offset", "return physical_block * block_size + offset;",
     "return physical_block * block_size - offset;", ["slot_examples"]),
    ("qsl_drops_running_sum", "query_start_loc[r + 1] = query_start_loc[r] + q_lens[r];",
     "query_start_loc[r + 1] = q_lens[r];", ["qsl"]),
    ("positions_off_by_one", "int64_t first_pos = (int64_t)seq_lens[r] - q_len;",
     "int64_t first_pos = (int64_t)seq_lens[r] - q_len + 1;", ["positions"]),
    ("kv_bytes_drops_factor_two", "return 2LL * num_layers", "return 1LL * num_layers",
     ["kv_bytes"]),
    ("score_drops_scale", "s[t] = scale * dot;", "s[t] = dot;", ["sdpa_decode"]),
    ("softmax_adds_epsilon", "double p = s[t] / l;", "double p = s[t] / (l + 1e-6);",
     ["sdpa_decode"]),
    ("gqa_wrong_kv_head", "h / group, num_kv_heads, head_dim, block_size, scale, s);\n            }\n            free(s);\n        }\n    }\n    return failed ? -2 : 0;\n}\n\n/* ---- Varlen",
     "h % num_kv_heads, num_kv_heads, head_dim, block_size, scale, s);\n            }\n            free(s);\n        }\n    }\n    return failed ? -2 : 0;\n}\n\n/* ---- Varlen", ["sdpa_decode"]),
    ("value_row_reversed_in_block",
     "const uint16_t* v = value_cache + ((phys * block_size + off) * num_kv_heads",
     "const uint16_t* v = value_cache + ((phys * block_size + (block_size - 1 - off)) * num_kv_heads",
     ["sdpa_decode"]),
    ("causal_limit_off_by_one", "context + i + 1,", "context + i,", ["sdpa_prefill"]),
    ("online_forgets_to_rescale_l", "l *= alpha;", "/* l not rescaled */", ["online"]),
    ("merge_drops_rescale", "L += l_parts[p] * exp(m_parts[p] - m);", "L += l_parts[p];",
     ["merge"]),
    ("writer_writes_past_the_pool",
     "if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;\n        int64_t block = slot / block_size;\n        int64_t offset",
     "if (slot < 0) continue;\n        int64_t block = slot / block_size;\n        int64_t offset",
     ["writer_pool_end"]),
    ("writer_shifts_offset", "int64_t offset = slot % block_size;\n        for",
     "int64_t offset = (slot + 1) % block_size;\n        for", ["writer"]),
    ("kernel_ids_transposed", "(int32_t)((int64_t)ids[i] * k + j)", "(int32_t)((int64_t)ids[i] + j * k)",
     ["kernel_blocks"]),
    ("kernel_ids_padding_kept", "ids[i] < 0 ? -1 :", "ids[i] < -1 ? -1 :", ["kernel_blocks_padding"]),
    ("e4m3_ties_away_from_zero", "if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;",
     "if (r >= 0.5) fl += 1.0;", ["e4m3_torch"]),
    ("e4m3_no_saturation", "if (a > 448.0) a = 448.0;", "/* no clamp */", ["e4m3_saturate"]),
    ("e4m3_subnormal_scale", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);",
     ["e4m3_decode"]),
    ("fp8_decode_ignores_v_scale", "(oracle_e4m3_decode(vr[x]) * v_scale)", "(oracle_e4m3_decode(vr[x]))",
     ["fp8_decode"]),
    ("xsplit_k_reverses_x", "* ORACLE_XSPLIT_X + d % ORACLE_XSPLIT_X;",
     "* ORACLE_XSPLIT_X + (ORACLE_XSPLIT_X - 1 - d % ORACLE_XSPLIT_X);", ["xsplit_layout"]),
    ("xsplit_v_reverses_offset", "* head_dim + d) * block_size + offset;",
     "* head_dim + d) * block_size + (block_size - 1 - offset);", ["xsplit_layout"]),
    ("xsplit_decode_drops_scale", "w[t] = scale * acc;", "w[t] = acc;", ["xsplit_decode"]),
    ("xsplit_decode_unnormalised", "double p = w[t] / total;", "double p = w[t];",
     ["xsplit_decode"]),
    ("xsplit8_k_uses_bf16_x", "* ORACLE_XSPLIT_X8 + d % ORACLE_XSPLIT_X8;",
     "* ORACLE_XSPLIT_X8 + d % ORACLE_XSPLIT_X;", ["xsplit8_writer"]),
    ("xsplit8_writer_skips_v_scale", "oracle_e4m3_encode(vf / v_scale);\n            }\n    }\n}\n\n/* Paged decode over e4m3 x-split",
     "oracle_e4m3_encode(vf);\n            }\n    }\n}\n\n/* Paged decode over e4m3 x-split", ["xsplit8_writer"]),
    ("fp8_prefill_ignores_k_scale", "(oracle_e4m3_decode(k[x]) * k_scale)", "(oracle_e4m3_decode(k[x]))",
     ["fp8_prefill"]),
    ("fp8_prefill_causal_off_by_one", "context + 1 + i,", "context + i,", ["fp8_prefill_rows"]),
    ("fp8_prefill_reads_kv_head_of_q_head", "h / group, num_kv_heads, head_dim, block_size, scale, k_scale,",
     "h % num_kv_heads, num_kv_heads, head_dim, block_size, scale, k_scale,", ["fp8_prefill"]),
    ("xsplit8_decode_unnormalised", "const double pw = w[t] / total;", "const double pw = w[t];",
     ["xsplit8_decode"]),
]

PINS = {
    "slot_examples": lambda o: pins.test_slot_examples_printed_on_pages(o),
    "qsl": lambda o: pins.test_query_start_loc_printed_on_pages(o),
    "positions": lambda o: pins.test_varlen_positions_of_mixed_batch(o),
    "kv_bytes": lambda o: pins.test_kv_bytes_formula_printed_on_pages(o),
    "sdpa_decode": lambda o: pins.test_decode_matches_torch_sdpa(o, 4, 2, 64, [25, 12, 37, 20], 16),
    "sdpa_decode_b32": lambda o: pins.test_decode_matches_torch_sdpa(o, 8, 2, 64, [31, 64, 70], 32),
    "kernel_blocks": lambda o: pins.test_kernel_blocks_printed_on_pages(o),
    "e4m3_torch": lambda o: pins.test_e4m3_encode_matches_torch_in_range(o),
    "e4m3_saturate": lambda o: pins.test_e4m3_encode_saturates_and_keeps_nan(o),
    "e4m3_decode": lambda o: pins.test_e4m3_codes_decode_like_torch(o),
    "fp8_decode": lambda o: pins.test_decode_fp8_equals_decode_of_dequantized_cache(o, 0.25, 4.0),
    "kernel_blocks_padding": lambda o: pins.test_kernel_blocks_identity_and_padding(o),
    "sdpa_prefill": lambda o: pins.test_prefill_matches_torch_sdpa_bottom_right_causal(o),
    "online": lambda o: pins.test_online_softmax_equals_direct(o, "block16"),
    "merge": lambda o: pins.test_partition_merge_equals_global_softmax(o),
    "writer": lambda o: pins.test_reshape_and_cache_scatter(o),
    "writer_pool_end": lambda o: pins.test_reshape_and_cache_skips_slots_past_the_pool(o),
    "xsplit_layout": lambda o: pins.test_xsplit_writer_places_elements_at_the_pages_shape(o, 2, 64, 16),
    "xsplit_decode": lambda o: pins.test_decode_xsplit_equals_decode_of_the_same_cache(
        o, 4, 2, 64, [25, 12, 37, 20], 16),
    "xsplit8_writer": lambda o: pins.test_xsplit_fp8_writer_is_a_permutation_of_the_token_major_fp8_writer(
        o, 0.013, 7.7),
    "fp8_prefill": lambda o: pins.test_prefill_fp8_equals_prefill_of_dequantized_cache(o, 0.5, 8.0),
    "fp8_prefill_rows": lambda o: pins.test_prefill_fp8_equals_prefill_of_dequantized_cache(o, 1.0, 1.0),
    "xsplit8_decode": lambda o: pins.test_decode_xsplit_fp8_equals_decode_fp8_of_the_same_cache(
        o, 4, 2, 64, [25, 12, 37, 20], 16),
}


def test_unplanted_copy_passes_every_pin(tmp_path):
    lib = oracle_pkg.build(src=SRC, out=str(tmp_path / "liboracle_copy.so"), force=True)
    o = oracle_pkg.Oracle(oracle_pkg.load(lib))
    for name, pin in PINS.items():
        pin(o)


@pytest.mark.parametrize("name,orig,planted,expect", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, orig, planted, expect):
    with open(SRC, encoding="utf-8") as f:
        text = f.read()
    assert text.count(orig) == 1, f"snippet for {name} must occur exactly once"
    src = tmp_path / "pa_oracle.c"
    src.write_text(text.replace(orig, planted), encoding="utf-8")
    hdr = os.path.join(os.path.dirname(SRC), "pa_oracle.h")
    (tmp_path / "pa_oracle.h").write_text(open(hdr, encoding="utf-8").read(), encoding="utf-8")
    lib = oracle_pkg.build(src=str(src), out=str(tmp_path / "libmutant.so"), force=True)
    o = oracle_pkg.Oracle(oracle_pkg.load(lib))
    for pin in expect:
        with pytest.raises(AssertionError):
            PINS[pin](o)
