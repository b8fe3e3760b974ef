"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them.

Each mutant is oracle.c with one textual change (an off-by-one in a mask, a
dropped scale, a wrong head mapping, a reversed index, a wrong merge weight),
compiled with gcc into a temporary library.  The pins of
``test_oracle_pins.py`` are run against it; at least one must fail.  Nothing
here touches a GPU.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement, occurrence index or None for all)
MUTANTS = [
    ("causal_off_by_one", "(j <= qpos)", "(j < qpos)", None),
    ("causal_dropped", "(j <= qpos) && ", "", None),
    ("window_off_by_one", "qpos - j <= window", "qpos - j < window", None),
    ("window_sign", "qpos - j <= window", "j - qpos <= window", None),
    ("scale_dropped", "double sj = sm_scale * dot;", "double sj = dot;", None),
    ("cap_inside_out", "logit_cap * tanh(sj / logit_cap)", "tanh(sj * logit_cap) / logit_cap", None),
    ("cap_before_scale", "double sj = sm_scale * dot;\n        if (logit_cap > 0.0)\n            sj = logit_cap * tanh(sj / logit_cap);",
     "double sj = dot;\n        if (logit_cap > 0.0)\n            sj = logit_cap * tanh(sj / logit_cap);\n        sj *= sm_scale;", None),
    ("lse_drops_max", "*lse = m + log(l);", "*lse = log(l);", None),
    ("no_normalise", "o[d] /= l;", "o[d] /= 1.0;", None),
    ("v_is_k", "o[d] += p * row_elem(vrow[j], d);", "o[d] += p * row_elem(krow[j], d);", None),
    ("gqa_modulo", "int hk = h / group;", "int hk = h % hkv;", None),
    ("extend_qpos_no_prefix", "p_len + i, sliding_window", "i, sliding_window", None),
    ("unified_qpos_no_prefix", "(long)prefix_lens[b] + i", "(long)i", None),
    ("extend_rows_reversed", "long te = qo_indptr[b] + e;", "long te = qo_indptr[b] + (e_len - 1 - e);", None),
    ("prefix_reversed", "long slot = kv_indices[kv_indptr[b] + j];\n            krow[j] = pool_row(k_buf, kv_fmt, k_scale, slot, k_buf_ss, k_buf_hs, hk);\n            vrow[j] = pool_row(v_buf, kv_fmt, v_scale, slot, v_buf_ss, v_buf_hs, hk);\n        }\n        for (long e = 0",
     "long slot = kv_indices[kv_indptr[b] + (p_len - 1 - j)];\n            krow[j] = pool_row(k_buf, kv_fmt, k_scale, slot, k_buf_ss, k_buf_hs, hk);\n            vrow[j] = pool_row(v_buf, kv_fmt, v_scale, slot, v_buf_ss, v_buf_hs, hk);\n        }\n        for (long e = 0", None),
    ("decode_qpos", "n_keys - 1, sliding_window", "n_keys - 2, sliding_window", None),
    ("merge_weight_uses_max", "double wa = exp(sa - s), wb = exp(sb - s);", "double wa = exp(sa - m), wb = exp(sb - m);", None),
    ("merge_lse_drops_max", "double s = m + log(exp(sa - m) + exp(sb - m));", "double s = log(exp(sa - m) + exp(sb - m));", None),
    ("merge_swapped", "wa * bf16_to_double(v_a[r * dv + d]) +\n                                wb * bf16_to_double(v_b[r * dv + d]);",
     "wb * bf16_to_double(v_a[r * dv + d]) +\n                                wa * bf16_to_double(v_b[r * dv + d]);", None),
    ("unified_extend_start_ignored", "extend_kv_indices[extend_start_loc[b] + e]", "extend_kv_indices[unified_kv_indptr[b] - prefix_kv_indptr[b] + e]", None),
    ("unified_indptr_drops_extend", "+ prefix_lens[b] + extend_seq_lens[b];", "+ prefix_lens[b];\n        unified_kv_indptr[b + 1] += extend_seq_lens[b] * (b > 0);", None),
    ("mask_ignored", "        if (mask_row)\n            visible = (mask_row[j] != 0) && (window <= 0 || qpos - j <= window);\n", "", None),
    ("mask_keeps_causal", "visible = (mask_row[j] != 0) && (window", "visible = (mask_row[j] != 0) && (j <= qpos) && (window", None),
    ("mask_row_stride", "custom_mask + mask_indptr[b] + i * n_keys : NULL;", "custom_mask + mask_indptr[b] + i : NULL;", None),
    ("sink_dropped", "    if (sink)\n        l += exp(*sink - m);\n", "", None),
    ("sink_sign", "l += exp(*sink - m);", "l += exp(m - *sink);", None),
    ("kvidx_start_ignored", "long start = kv_start_idx ? (long)(int32_t)kv_start_idx[b] : 0;", "long start = 0;", None),
    ("kvidx_row_is_batch_index", "long row = (long)req_pool_indices[b] * stride;", "long row = (long)b * stride;", None),
    ("kvidx_len_minus_start", "for (long j = 0; j < (long)(int32_t)paged_kernel_lens[b]; ++j)",
     "for (long j = 0; j < (long)(int32_t)paged_kernel_lens[b] - start; ++j)", None),
    ("kvidx_segment_reversed", "kv_indices[kv_indptr[b] + j] = req_to_token[row + start + j];",
     "kv_indices[kv_indptr[b + 1] - 1 - j] = req_to_token[row + start + j];", None),
    ("setkv_slot_is_token", "long slot = (long)cache_loc[t];", "long slot = t;", None),
    ("setkv_heads_reversed", "k[t * k_ts + (long)h * k_hs + d];", "k[t * k_ts + (long)(hkv - 1 - h) * k_hs + d];", None),
    ("setkv_v_from_k", "v[t * v_ts + (long)h * v_hs + d];", "k[t * k_ts + (long)h * k_hs + d];", None),
    ("fp8_e4m3_bias", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", None),
    ("fp8_e4m3_subnormal", "ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)", None),
    ("fp8_e5m2_bias", "ldexp(1.0 + m / 4.0, e - 15)", "ldexp(1.0 + m / 4.0, e - 16)", None),
    ("fp8_ties_to_odd", "(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)", None),
    ("fp8_scale_dropped", "r.fmt) * r.scale;", "r.fmt);", None),
    ("fp8_kv_scales_swapped", "pool_row(k_buf, kv_fmt, k_scale,", "pool_row(k_buf, kv_fmt, v_scale,", None),
    ("fp8_write_no_divide", "oracle_fp8_code(x / k_scale, fmt)", "oracle_fp8_code(x, fmt)", None),
    ("paged_offset_dropped", "kv_indices[kv_indptr[b] + j / page_size] * page_size +\n                (int32_t)(j % page_size);",
     "kv_indices[kv_indptr[b] + j / page_size] * page_size;", None),
    ("paged_last_page_len_ignored", "(pages - 1) * page_size + kv_last_page_len[b] : 0;", "(pages - 1) * page_size + 1 : 0;", None),
    ("paged_page_not_scaled", "kv_indices[kv_indptr[b] + j / page_size] * page_size +", "kv_indices[kv_indptr[b] + j / page_size] +", None),
    ("sink_in_values", "    if (sink)\n        l += exp(*sink - m);\n", "    if (sink) {\n        l += exp(*sink - m);\n        for (int d = 0; d < lv; ++d) o[d] += exp(*sink - m);\n    }\n", None),
]

# The pins, cheapest first; a mutant is caught by the first one that fails.
BATTERY = [
    lambda: pins.test_unified_indices_hand_fixture(),
    lambda: pins.test_merge_closed_forms(),
    lambda: pins.test_merge_weights_are_softmax_of_lse(),
    lambda: pins.test_no_prefix_is_torch_causal_sdpa(64, 64, 4, 2),
    lambda: pins.test_no_prefix_window_is_sdpa_band_mask(),
    lambda: pins.test_matches_dense_library_formulation(2.5, 40, 4),
    lambda: pins.test_matches_dense_library_formulation(0.0, 9, 3),
    lambda: pins.test_gqa_head_mapping(),
    lambda: pins.test_cap_two_key_closed_form(),
    lambda: pins.test_one_and_two_visible_keys_closed_forms(),
    lambda: pins.test_decode_equals_extend_of_last_token(),
    lambda: pins.test_decode_window_keeps_last_w_plus_one_keys(),
    lambda: pins.test_two_stage_equals_unified(),
    lambda: pins.test_unified_indices_are_per_sequence_concatenation(0),
    lambda: pins.test_merge_of_two_key_halves_equals_attention_over_all(),
    lambda: pins.test_custom_mask_matches_dense_formulation(0.0, -1, 1),
    lambda: pins.test_causal_pattern_mask_equals_no_mask(),
    lambda: pins.test_sinks_match_an_extra_zero_valued_key(-1),
    lambda: pins.test_sink_with_one_visible_key_closed_form(),
    lambda: pins.test_kv_indices_hand_fixture(),
    lambda: pins.test_set_kv_buffer_hand_fixture(),
    lambda: pins.test_kv_indices_are_row_slices(0),
    lambda: pins.test_set_kv_buffer_matches_index_copy(3, 128, 96, False),
    lambda: pins.test_fp8_code_values_match_torch(*pins.FP8[0]),
    lambda: pins.test_fp8_code_values_match_torch(*pins.FP8[1]),
    lambda: pins.test_fp8_rounding_matches_torch_in_range(*pins.FP8[0]),
    lambda: pins.test_fp8_write_matches_torch_quantization(),
    lambda: pins.test_fp8_pool_attention_equals_bf16_pool_of_its_values(pins.oracle.KV_E4M3),
    lambda: pins.test_paged_indices_hand_fixture(),
    lambda: pins.test_paged_indices_are_page_blocks(16),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation {name}: pattern not found in oracle.c"
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-w",
                    "-o", str(so), str(c), "-lm"], check=True)
    return str(so)


def test_unmutated_copy_passes_battery(tmp_path):
    """Control: the battery passes on an unmodified rebuild."""
    so = _build_mutant(tmp_path, "control", "#include <math.h>", "#include <math.h>")
    with oracle.use_library(so):
        for check in BATTERY:
            check()


@pytest.mark.parametrize("name,old,new,_", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, _):
    so = _build_mutant(tmp_path, name, old, new)
    with oracle.use_library(so):
        for check in BATTERY:
            try:
                check()
            except Exception:
                return  # caught
    pytest.fail(f"no pin caught the planted mistake {name!r}")
