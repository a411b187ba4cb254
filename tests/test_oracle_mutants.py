"""Plant plausible mistakes in a copy of the oracle and check the pins catch them.

Each mutant is the oracle's C source with one edit (a dropped term, a wrong sign
or index, a transposed operand, a wrong tie order ...), compiled with gcc into a
temporary directory.  The pins of test_oracle_pins.py are then run against it;
at least one must fail.  This runs on the CPU only.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "lora_oracle.c")

MUTANTS = {
    "drop_scale": ("yo[o + m] += scales[s] * acc;", "yo[o + m] += acc;"),
    "wrong_sign": ("yo[o + m] += scales[s] * acc;", "yo[o + m] -= scales[s] * acc;"),
    "drop_slice_offset": ("yo[o + m] += scales[s] * acc;", "yo[m] += scales[s] * acc;"),
    "transposed_B": ("bf16_value(b[(int64_t)m * r + j])", "bf16_value(b[(int64_t)j * di + m])"),
    "reversed_x": ("for (int32_t c = 0; c < k; ++c) acc += bf16_value(xt[c]) * bf16_value(a[(int64_t)j * k + c]);\n                xa[j] = acc;",
                   "for (int32_t c = 0; c < k; ++c) acc += bf16_value(xt[k - 1 - c]) * bf16_value(a[(int64_t)j * k + c]);\n                xa[j] = acc;"),
    "drop_y_in": ("yo[m] = y_in ? bf16_value(y_in[(int64_t)t * ldy + m]) : 0.0;", "yo[m] = 0.0;"),
    "unstable_ties": ("return a->t < b->t ? -1 : (a->t > b->t ? 1 : 0);", "return a->t > b->t ? -1 : (a->t < b->t ? 1 : 0);"),
    "offsets_off_by_one": ("c += (key[t] < b);", "c += (key[t] <= b);"),
    "no_adapter_bucket_first": ("key[t] = S;\n            if (s != -1)", "key[t] = -1;\n            if (s != -1)"),
    "active_keeps_rank0": ("if (count > 0 && ranks[s] > 0) active", "if (count > 0) active"),
    "rslora_without_sqrt": ("adapter_scale * alpha / sqrt((double)rank)", "adapter_scale * alpha / (double)rank"),
    "alpha_zero_not_special": ("if (alpha == 0.0 || rank <= 0) return adapter_scale;", "if (rank <= 0) return adapter_scale;"),
    "ties_away_from_zero": ("q = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "q = fl + 1.0;"),
    "rank_loop_short": ("for (int32_t j = 0; j < r; ++j) {\n                double acc = 0.0;", "for (int32_t j = 0; j + 1 < r; ++j) {\n                double acc = 0.0;"),
    "e4m3_wrong_bias": ("v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);", "v = (1.0 + m / 8.0) * ldexp(1.0, e - 8);"),
    "e4m3_no_subnormals": ("if (e == 0) v = m * ldexp(1.0, -9);", "if (e == 0) v = (1.0 + m / 8.0) * ldexp(1.0, -7);"),
    "fp8_x_not_quantized": ("xq[c] = oracle_e4m3_to_double(oracle_e4m3_round(bf16_value(x[(int64_t)t * ldx + c])));",
                            "xq[c] = bf16_value(x[(int64_t)t * ldx + c]);"),
    "e4m3_ties_to_odd": ("(c & 1) == 0 && (best & 1) == 1", "(c & 1) == 1 && (best & 1) == 0"),
    "moe_A_offset_uses_d": ("A[(int64_t)s * n_slices + i] + (int64_t)e * k * r;",
                            "A[(int64_t)s * n_slices + i] + (int64_t)e * di * r;"),
    "moe_B_offset_uses_k": ("B[(int64_t)s * n_slices + i] + (int64_t)e * di * r;",
                            "B[(int64_t)s * n_slices + i] + (int64_t)e * k * r;"),
    "moe_x_row_per_pair": ("(int64_t)(x_per_token ? t : p) * ldx", "(int64_t)p * ldx"),
    "moe_ignores_expert": ("int32_t e = expert_ids[p];", "int32_t e = 0;"),
    "moe_expert_from_token": ("int32_t e = expert_ids[p];", "int32_t e = expert_ids[t];"),
}

PINS = [
    lambda: pins.test_index_brute_force_all_tiny_inputs((8, 8)),
    lambda: pins.test_index_brute_force_all_tiny_inputs((0, 16)),
    lambda: pins.test_index_matches_library_stable_sort(1),
    pins.test_branch_matches_library_matmul,
    pins.test_merged_weight_identity,
    pins.test_orientation_matches_printed_shapes,
    pins.test_closed_form_one_hot_rank1,
    pins.test_zero_B_and_no_adapter_rows_are_unchanged,
    pins.test_rslora_versus_standard_scale,
    pins.test_scale_values_printed_on_pages,
    pins.test_premultiplied_scale_equals_runtime_scale,
    pins.test_rank_concatenation_identity,
    pins.test_mac_count_matches_pages,
    pins.test_rank0_slot_and_out_of_range_slot,
    pins.test_round_bf16_against_brute_force,
    pins.test_e4m3_decode_matches_library_on_every_code,
    pins.test_e4m3_round_matches_library_clamp_and_convert,
    pins.test_e4m3_premultiply_matches_pages_expression,
    pins.test_fp8_branch_equals_bf16_branch_on_decoded_values,
    lambda: pins.test_moe_one_hot_at_the_pages_expert_offset(True),
    lambda: pins.test_moe_one_hot_at_the_pages_expert_offset(False),
    pins.test_moe_single_expert_reduces_to_dense_branch,
    pins.test_moe_choice_order_and_shared_rows,
    pins.test_moe_out_of_range_ids_and_pair_slots,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(mutated)
    so_path = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(so_path), str(c_path), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.configure(ctypes.CDLL(str(so_path))))
    failures = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin caught mutant {name}"


# The speculative-decode index is a thin rule in oracle/__init__.py (token order
# of sequences of tps tokens); plant the two plausible slips in that rule.
SEQ_MUTANTS = {
    # tokens interleaved across sequences instead of sequence-major
    "tiled_tokens": lambda seq, tps, S, ranks: oracle.build_index(
        np.tile(np.asarray(seq, np.int32), int(tps)), S, ranks),
    # the sequence index reused without expanding it to tokens
    "not_expanded": lambda seq, tps, S, ranks: oracle.build_index(np.asarray(seq, np.int32), S, ranks),
}


@pytest.mark.parametrize("name", sorted(SEQ_MUTANTS))
def test_pins_catch_planted_speculative_index_mistake(name, monkeypatch):
    monkeypatch.setattr(oracle, "build_index_seq", SEQ_MUTANTS[name])
    with pytest.raises(AssertionError):
        pins.test_speculative_index_matches_pages_expansion(2, 4)


# Activated-LoRA enablement is a thin rule in oracle/__init__.py; plant the
# plausible slips in it.
ACT_MUTANTS = {
    # the adapter starts one token late (strict comparison)
    "strict_start": lambda seq, pos, slot, start: np.where(
        np.asarray(pos) > np.asarray(start)[np.asarray(seq)], np.asarray(slot)[np.asarray(seq)], -1).astype(np.int32),
    # the adapter applies before the invocation point instead of after it
    "reversed": lambda seq, pos, slot, start: np.where(
        np.asarray(pos) < np.asarray(start)[np.asarray(seq)], np.asarray(slot)[np.asarray(seq)], -1).astype(np.int32),
    # the invocation start ignored
    "always_on": lambda seq, pos, slot, start: np.asarray(slot)[np.asarray(seq)].astype(np.int32),
}


@pytest.mark.parametrize("name", sorted(ACT_MUTANTS))
def test_pins_catch_planted_activation_mistake(name, monkeypatch):
    monkeypatch.setattr(oracle, "activated_token_slots", ACT_MUTANTS[name])
    with pytest.raises((AssertionError, IndexError)):
        pins.test_activated_slots_hand_worked()
