"""Each plausible mistake, planted in a copy of the oracle's C source and
compiled on the CPU, must fail at least one independent pin (the digest test,
which compares the oracle with its own earlier output, is not counted)."""
import inspect

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_fake_quant as qpins
from tests import test_oracle_floors as flpins
from tests import test_oracle_fp8 as fpins
from tests import test_oracle_variants as vpins
from tests import test_scorer_oracle as spins

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("tie_to_odd", "(d == best_d && (m % 2) == 0 && (best % 2) != 0)",
     "(d == best_d && (m % 2) != 0 && (best % 2) == 0)"),
    ("tie_toward_lower_code", " || (d == best_d && (m % 2) == 0 && (best % 2) != 0)", ""),
    ("keep_negative_zero", "int neg = (z[i] < 0.0f) && (m != 0);", "int neg = (z[i] < 0.0f);"),
    ("nibble_order_swapped", "(uint8_t)(n2[2 * j] | (n2[2 * j + 1] << 4))",
     "(uint8_t)(n2[2 * j + 1] | (n2[2 * j] << 4))"),
    ("exponent_floor_not_ceil", "+ ((bits & 0x7fffffu) != 0u ? 1 : 0)", "+ 0"),
    ("amax_over_4", "float t = amax / 6.0f;", "float t = amax / 4.0f;"),
    ("large_stage1_amax_floor", "STAGE1_AMAX_FLOOR = 1.17549435082228750797e-38f",
     "STAGE1_AMAX_FLOOR = 1e-10f"),
    ("large_stage2_quotient_floor", "STAGE2_QUOT_FLOOR = 1.17549435082228750797e-38f",
     "STAGE2_QUOT_FLOOR = 1e-10f"),
    ("single_stage", "int e2 = oracle_quant_group_floors(u, s2_amax, s2_quot, n2);",
     "int e2 = e1; memcpy(n2, n1, GROUP);"),
    ("scale_bias_off_by_one", "double scale = ldexp(1.0, e - 127);",
     "double scale = ldexp(1.0, e - 128);"),
    ("amax_signed", "float a = fabsf(z[i]);", "float a = z[i];"),
    ("exp_bytes_reversed", "exp4[g] = (uint8_t)e2;", "exp4[3 - g] = (uint8_t)e2;"),
    ("mean_over_64", "float ms = sum / 128.0f;", "float ms = sum / 64.0f;"),
    ("eps_outside_sqrt", "float den = ms + eps;\n  float root = sqrtf(den);",
     "float den = ms;\n  float root = sqrtf(den) + eps;"),
    ("gamma_dropped", "float xg = xr * bf16_to_f32(gamma[i]);", "float xg = xr;"),
    ("no_reciprocal", "float r = 1.0f / root;", "float r = root;"),
    ("rope_sign", "float na = ac - bs;", "float na = ac + bs;"),
    ("rope_cos_sin_swapped", "float c = cos_row[i];\n    float s = sin_row[i];",
     "float c = sin_row[i];\n    float s = cos_row[i];"),
    ("rope_neox_partner_half_head", "ib = i + ROPE_DIM / 2;", "ib = i + HEAD_DIM / 2;"),
    ("rope_interleaved_table_index", "float c = cos_row[i];",
     "float c = cos_row[rope_style == ORACLE_ROPE_NEOX ? i : (2 * i) % 32];"),
    ("slot_record_interleaved",
     "memcpy(page + o * PAYLOAD_BYTES, r, PAYLOAD_BYTES);\n"
     "    memcpy(page + KV_BLOCK * PAYLOAD_BYTES + o * EXP_BYTES, r + PAYLOAD_BYTES, EXP_BYTES);",
     "memcpy(page + o * 68, r, PAYLOAD_BYTES);\n"
     "    memcpy(page + o * 68 + PAYLOAD_BYTES, r + PAYLOAD_BYTES, EXP_BYTES);"),
    ("slot_zero_skipped", "if (slot < 0) continue;", "if (slot <= 0) continue;"),
    ("weights_scale_no_sqrt_of_heads",
     "double wscale = 1.0 / sqrt((double)num_heads * (double)HEAD_DIM);",
     "double wscale = 1.0 / ((double)num_heads * sqrt((double)HEAD_DIM));"),
    ("bf16_truncate", "if (d_lo < d_hi)\n    pick = lo;", "if (1)\n    pick = lo;"),
    ("bf16_ties_up", "pick = ((lo >> 16) & 1u) ? hi : lo;", "pick = hi;"),
    ("q_rope_skipped",
     "      oracle_rope_row(y, cos_cache + pos * (ROPE_DIM / 2),\n"
     "                      sin_cache + pos * (ROPE_DIM / 2), rope_style);\n", ""),
    ("scorer_no_relu", "if (dot > 0.0) acc += (double)weights[r] * dot;",
     "acc += (double)weights[r] * dot;"),
    ("scorer_weight_dropped", "if (dot > 0.0) acc += (double)weights[r] * dot;",
     "if (dot > 0.0) acc += dot;"),
    ("scorer_slot_offset_off_by_one", "int64_t o = s % KV_BLOCK;\n      key_values(",
     "int64_t o = (s + 1) % KV_BLOCK;\n      key_values("),
    ("scorer_key_group_exponent", "int ke = pg[KV_BLOCK * PAYLOAD_BYTES + o * EXP_BYTES + d / GROUP];",
     "int ke = pg[KV_BLOCK * PAYLOAD_BYTES + o * EXP_BYTES + (d / GROUP + 1) % 4];"),
    ("scorer_key_nibble_swap", "uint8_t knib = (d % 2) ? (kbyte >> 4) : (kbyte & 15);",
     "uint8_t knib = (d % 2) ? (kbyte & 15) : (kbyte >> 4);"),
    ("scorer_query_exponent_bias", "qv[d] = dequant_d(qnib, q_scale[r * EXP_BYTES + d / GROUP]);",
     "qv[d] = dequant_d(qnib, q_scale[r * EXP_BYTES + d / GROUP] + 1);"),
    ("scorer_padding_zero", "      if (s >= ctx) {\n        *out = -INFINITY;",
     "      if (s >= ctx) {\n        *out = 0.0f;"),
    ("k_rope_skipped",
     "    oracle_rope_row(y, cos_cache + rope_pos * (ROPE_DIM / 2),\n"
     "                    sin_cache + rope_pos * (ROPE_DIM / 2), rope_style);\n", ""),
    ("hadamard_sign", "x[j + h] = a - b;", "x[j + h] = b - a;"),
    ("hadamard_norm_over_128", "(float)(1.0 / sqrt((double)HEAD_DIM))",
     "(float)(1.0 / (double)HEAD_DIM)"),
    ("hadamard_stage_dropped", "for (int h = 1; h < HEAD_DIM; h *= 2)",
     "for (int h = 1; h < HEAD_DIM / 2; h *= 2)"),
    ("hadamard_pair_distance", "float a = x[j], b = x[j + h];",
     "float a = x[j], b = x[(j + h + 1) % HEAD_DIM];"),
    ("compress_divides", "int64_t rope_pos = pos - pos % compress_ratio;",
     "int64_t rope_pos = pos / compress_ratio;"),
    ("compress_ignored", "int64_t rope_pos = pos - pos % compress_ratio;",
     "int64_t rope_pos = pos;"),
    ("k_hadamard_skipped", "    if (hadamard) oracle_hadamard_row(y);\n    uint8_t* r = rec",
     "    uint8_t* r = rec"),
    ("fp8_max_240", "float t = amax / 448.0f;", "float t = amax / 240.0f;"),
    ("fp8_scale_floor_not_ceil", "+ (int)((bits & 0x7fffffu) != 0u);", "+ 0;"),
    ("fp8_ties_down", "if (d < best_d || (d == best_d && (c % 2) == 0 && (best % 2) != 0)) {",
     "if (d < best_d) {"),
    ("fp8_sign_dropped", "return (uint8_t)(best | (signbit(v) ? 0x80 : 0));",
     "return (uint8_t)best;"),
    ("fp8_weight_scale_not_folded",
     "folded = ldexp(1.0, fp8_quant_row(y, q_out + r * HEAD_DIM) - 127);",
     "fp8_quant_row(y, q_out + r * HEAD_DIM);"),
    ("fp8_scale_slot_interleaved", "memcpy(page + KV_BLOCK * HEAD_DIM + o * 4, r + HEAD_DIM, 4);",
     "memcpy(page + KV_BLOCK * HEAD_DIM + (63 - o) * 4, r + HEAD_DIM, 4);"),
    ("fq16_amax_over_4", "float t16 = amax16 / 6.0f;", "float t16 = amax16 / 4.0f;"),
    ("fq16_scale_not_e4m3", "float sc = oracle_e4m3_to_f32(oracle_f32_to_e4m3(t16));",
     "float sc = t16;"),
    ("fq16_keep_negative_zero", "out[i] = (float)((v < 0.0f && m != 0) ? -d : d);",
     "out[i] = (float)((v < 0.0f) ? -d : d);"),
    ("fq16_multiply_not_divide", "float v = z[i] / sc;", "float v = z[i] * sc;"),
    ("fq_rope_skipped",
     "    oracle_rope_row(y, cos_cache + pos * (ROPE_DIM / 2),\n"
     "                    sin_cache + pos * (ROPE_DIM / 2), rope_style);\n"
     "    oracle_fake_quant_row", "    oracle_fake_quant_row"),
    ("prefill_range_end_inclusive", "if (s < ks[t] || s >= ke[t]) {",
     "if (s < ks[t] || s > ke[t]) {"),
    ("prefill_key_page_shifted", "key_values(kv_cache + (s / KV_BLOCK) * PAGE_BYTES, s % KV_BLOCK, kv);",
     "key_values(kv_cache + ((s + 64) / KV_BLOCK % 2) * PAGE_BYTES, s % KV_BLOCK, kv);"),
    ("q_hadamard_skipped", "      if (hadamard) oracle_hadamard_row(y);\n      double folded",
     "      double folded"),
]

# Independent pins, cheapest first.
PINS = [
    pins.test_golden_e2m1_values,
    pins.test_golden_pack_layout,
    pins.test_all_zero_group,
    pins.test_rmsnorm_constant_row_closed_form,
    pins.test_rmsnorm_midpoint_key_row,
    pins.test_rmsnorm_eps_inside_sqrt,
    pins.test_rope_identity_and_quarter_turn,
    pins.test_rope_single_pair_and_general,
    pins.test_cache_store_placement_and_skip,
    pins.test_out_of_range_rows_are_skipped,
    pins.test_golden_midpoint_key_slot,
    pins.test_golden_tiny_query_midpoints,
    pins.test_k_op_closed_form_composition,
    pins.test_q_op_closed_form_composition,
    pins.test_weights_closed_form,
    spins.test_single_element_closed_form,
    spins.test_heads_weighted_relu_sum,
    spins.test_group_exponents_scale_the_score,
    spins.test_page_indirection_and_sequences,
    spins.test_bad_page_reported,
    spins.test_random_case_exact_rational,
    spins.test_prefill_single_element_closed_form,
    spins.test_prefill_ranges_and_exact_values,
    flpins.test_tiny_groups_two_stage_exact,
    vpins.test_hadamard_one_hot_rows,
    vpins.test_hadamard_small_integers_exact,
    vpins.test_query_rotation_sign_pattern,
    vpins.test_key_rotation_sign_pattern,
    vpins.test_compress_ratio_uses_group_first_position,
    fpins.test_encode_saturates_above_448,
    fpins.test_all_zero_row_floor,
    fpins.test_key_slot_closed_form,
    fpins.test_query_weight_folds_scale,
    fpins.test_decode_all_codes_match_torch,
    fpins.test_encode_matches_torch_in_range,
    fpins.test_row_exponent_exact,
    qpins.test_mode1_midpoints_closed_form,
    qpins.test_mode1_tiny_group_is_zero_and_saturation,
    qpins.test_rope_then_fake_quant_at_position_zero,
    qpins.test_mode1_per16_e4m3_exact,
    qpins.test_mode0_is_per32_ue8m0_exact,
    pins.test_two_stage_invariants,
    pins.test_group_quant_exact_rational,
    pins.test_exponent_exhaustive_bf16,
    pins.test_bf16_rounding_matches_torch,
    pins.test_rmsnorm_random_rows_vs_fp64,
    pins.test_codes_exhaustive_bf16,
]


def _run(fn):
    params = inspect.signature(fn).parameters
    if "style" in params:
        for s in (0, 1):
            fn(style=s)
    elif "ratio" in params:
        for r in (2, 4):
            fn(ratio=r)
    else:
        fn()


def test_unmutated_oracle_passes_all_pins():
    for fn in PINS:
        _run(fn)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    L = oracle.compile_variant(src.replace(old, new), str(tmp_path))
    caught = None
    with oracle.use_variant(L):
        for fn in PINS:
            try:
                _run(fn)
            except AssertionError:
                caught = fn.__name__
                break
    assert caught is not None, f"mutant {name} passed every pin"
