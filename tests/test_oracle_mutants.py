"""The pins catch plausible mistakes: each test plants one mistake in a copy
of the oracle's C source, compiles it on the CPU, and requires that at least
one pin fails.  The real oracle is never modified."""
import os
import subprocess

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ts_oracle.c")

MUTANTS = {
    "tie_order_reversed": ("return (a->index < b->index) ? -1 : (a->index > b->index);",
                           "return (a->index > b->index) ? -1 : (a->index < b->index);"),
    "temperature_dropped": ("exp((scratch[j].value - m) / (double)temp)",
                            "exp((scratch[j].value - m))"),
    "max_sign_flipped": ("exp((scratch[j].value - m) / (double)temp)",
                         "exp((m - scratch[j].value) / (double)temp)"),
    "nucleus_strict": ("if (cum >= (double)top_p) {", "if (cum > (double)top_p) {"),
    "draw_non_strict": ("if (pick < 0 && c > u) pick = j;", "if (pick < 0 && c >= u) pick = j;"),
    "philox_wrong_product": ("uint64_t y0 = hi1 ^ x1 ^ k0;", "uint64_t y0 = hi0 ^ x1 ^ k0;"),
    "philox_no_key_bump": ("    k0 += W0;\n", "\n"),
    "philox_9_rounds": ("for (int round = 0; round < 10; ++round)",
                        "for (int round = 0; round < 9; ++round)"),
    "uniform_wrong_word": ("return (uint32_t)(out[0] >> 40);", "return (uint32_t)(out[1] >> 40);"),
    "counter_swapped": ("{(uint64_t)step, (uint64_t)(int64_t)codebook, 0, 0}",
                        "{(uint64_t)(int64_t)codebook, (uint64_t)step, 0, 0}"),
    "no_cap_clamp": ("  if (k > cap) k = cap;\n", "\n"),
    "no_topk_zero_rule": ("int64_t k = top_k > 0 ? top_k : vocab;",
                          "int64_t k = top_k > 0 ? top_k : 1;"),
    "eos_flag_inverted": ("(uint8_t)(b->eos_id[r] >= 0 && id == b->eos_id[r])",
                          "(uint8_t)(b->eos_id[r] >= 0 && id != b->eos_id[r])"),
    "greedy_only_negative": ("if (temp <= 0.0f || k_eff == 1) {", "if (temp < 0.0f || k_eff == 1) {"),
    "nucleus_mass_off_by_one": ("for (int j = 0; j < n_p; ++j) s_p += qbuf[j];",
                                "for (int j = 0; j + 1 < n_p; ++j) s_p += qbuf[j];"),
    "pinf_accepted": ("if (isnan(v) || v == INFINITY) bad_value = 1;",
                      "if (isnan(v)) bad_value = 1;"),
    "bf16_widen_wrong": ("uint32_t bits = (uint32_t)b << 16;", "uint32_t bits = (uint32_t)b << 15;"),
    "cap_upper_4095": ("if (requested < 32 || requested > 4096) return -1;",
                       "if (requested < 32 || requested > 2048) return -1;"),
    "offset_check_dropped": ("off > b->logits_len - (int64_t)vocab)", "off > b->logits_len)"),
    # the finished-stream rule
    "finish_length_before_stop": (
        "  if (b->stop_step && b->stop_step[stream] >= 0 && b->stop_step[stream] < t) return 1;\n"
        "  if (b->max_steps && t >= b->max_steps[stream]) return 2;",
        "  if (b->max_steps && t >= b->max_steps[stream]) return 2;\n"
        "  if (b->stop_step && b->stop_step[stream] >= 0 && b->stop_step[stream] < t) return 1;"),
    "finish_stop_recorded_late": ("if (b->stop_step) b->stop_step[stream] = b->step[stream];",
                                  "if (b->stop_step) b->stop_step[stream] = b->step[stream] + 1;"),
    "finish_cap_exclusive": ("if (b->max_steps && t >= b->max_steps[stream]) return 2;",
                             "if (b->max_steps && t > b->max_steps[stream]) return 2;"),
    # the repetition penalty
    "penalty_on_duplicates": ("          if (!seen) hist[n_hist++] = x;", "          hist[n_hist++] = x;"),
    "penalty_divides_negatives": ("float pen = f > 0.0f ? f / theta : f * theta;",
                                  "float pen = f / theta;"),
    "penalty_not_rounded": ("  if (dtype == 1) pen = round_to_bf16(pen);", ""),
    "penalty_ring_slot_late": ("int64_t j = ((t % b->hist_len) + b->hist_len) % b->hist_len;",
                               "int64_t j = ((t + 1) % b->hist_len + b->hist_len) % b->hist_len;"),
    # the LM head
    "lm_head_wrong_head": ("const int64_t hoff = head_offsets[r % n_heads];",
                           "const int64_t hoff = head_offsets[(r / n_heads) % n_heads];"),
    "lm_head_transposed": ("load_value(1, weights, w0 + k);",
                           "load_value(1, weights, hoff + (int64_t)k * vr + v);"),
    "lm_head_float_sum": ("      double acc = 0.0;\n      for (int32_t k = 0; k < dim; ++k)\n",
                          "      float acc = 0.0f;\n      for (int32_t k = 0; k < dim; ++k)\n"),
    "lm_head_no_alignment_rule": ("hoff >= 0 && hoff % 8 == 0 && hoff <=", "hoff >= 0 && hoff <="),
    "lm_head_bound_one_row_short": ("hoff <= weights_len - (int64_t)vr * dim;",
                                    "hoff <= weights_len - (int64_t)(vr - 1) * dim;"),
    "lm_head_next_hidden_row": ("const int64_t h0 = r * (int64_t)dim;",
                                "const int64_t h0 = ((r + 1) % n_rows) * (int64_t)dim;"),
    # the boundary margin that excuses rows from the bit-exact rule
    "margin_draw_unnormalised": ("double d = fabs(c - u);", "double d = fabs(cum - u);"),
    "margin_cut_exclusive_prefix": ("double d = fabs(cum - (double)top_p);",
                                    "double d = fabs(cum - qbuf[n - 1] - (double)top_p);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "ts_oracle_mutant.c"
    mutated.write_text(src.replace(old, new), encoding="utf-8")
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(lib),
                           str(mutated), "-lm", "-lpthread"])
    mut = oracle.Oracle(str(lib))
    caught = []
    for pin in PINS:
        try:
            pin(mut)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin detects mutant {name}"
