"""Strength of the oracle's pins: plant a plausible mistake in a copy of the
oracle source (on the CPU), rebuild it, and check that at least one pin from
``test_oracle_pins`` fails against the broken copy, while all of them pass
against the real one."""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gqa_oracle.c")

PIN_BATTERY = [
    pins.test_head_map_worked_example,
    pins.test_mha_special_case_matches_library_attention,
    pins.test_mqa_special_case_matches_shared_kv_einsum,
    lambda: pins.test_general_gqa_matches_library_attention(8, 2),
    pins.test_identical_keys_give_plain_mean,
    pins.test_zero_scale_gives_plain_mean,
    pins.test_length_one_returns_first_value_row,
    pins.test_dominant_logit_selects_its_value,
    pins.test_softmax_weights_sum_to_one,
    pins.test_poisoned_tail_is_never_read,
    pins.test_empty_and_overlong_lengths,
    pins.test_brute_force_high_precision,
    pins.test_kv_append_oracle_places_rows_and_increments,
    pins.test_append_then_attend_includes_new_token,
    pins.test_meanpool_identity_when_groups_equal_heads,
    pins.test_meanpool_single_group_is_mean_of_all_heads,
    pins.test_meanpool_is_the_group_mean_of_projections,
    pins.test_multi_token_single_token_is_the_decode_oracle,
    pins.test_multi_token_is_causal_prefix_attention,
    pins.test_multi_token_sees_nothing_before_the_cache,
    pins.test_multi_token_brute_force,
    pins.test_projection_with_identity_weights_slices_x,
    pins.test_projection_of_mean_pooled_weights_is_the_group_mean,
    pins.test_projection_matches_the_blog_einsums,
    pins.test_projection_brute_force,
    pins.test_e4m3_decode_table_matches_torch,
    pins.test_e4m3_encode_is_nearest_even_and_saturates,
    pins.test_fp8_attention_is_attention_on_the_dequantized_cache,
    pins.test_fp8_append_quantizes_and_places_the_row,
]

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("interleaved head->group map",
     "off[(size_t)b * H + (size_t)g * n_rep + r]", "off[(size_t)b * H + (size_t)r * G + g]"),
    ("no max subtraction", "w[n] = exp(w[n] - m);", "w[n] = exp(w[n]);"),
    ("scale dropped", "w[n] = dot * scale;", "w[n] = dot;"),
    ("reads one position past L", "int b = (int)(bh / H);\n        int L = clamp_len(seq_lens[b], Nmax);",
     "int b = (int)(bh / H);\n        int L = clamp_len(seq_lens[b] + 1, Nmax);"),
    ("softmax not normalised", "for (int n = 0; n < L; ++n) w[n] /= z;", "(void)z;"),
    ("K used in place of V", "o[i] += w[n] * load_value(v, kv_off[bh]", "o[i] += w[n] * load_value(k, kv_off[bh]"),
    ("several tokens: a token also sees the next one", "int vis = L - T + 1 + t;", "int vis = L - T + 2 + t;"),
    ("several tokens: views in reverse token order", "int vis = L - T + 1 + t;", "int vis = L - t;"),
    ("several tokens: every token reads token 0's query", "head_weights(q, k, (size_t)bth * d,",
     "head_weights(q, k, ((size_t)b * T * H + h) * d,"),
    ("several tokens: K used in place of V", "o[i] += w[n] * load_value(v, kvo", "o[i] += w[n] * load_value(k, kvo"),
    ("e4m3: exponent bias 8", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3: ties away from zero", "(err == best_err && (c & 1) == 0 && (best & 1) == 1)", "(err == best_err && c > best)"),
    ("fp8 append ignores the scale", "k_cache[dst + i] = e4m3_encode(kx / k_scale[g]);",
     "k_cache[dst + i] = e4m3_encode(kx);"),
    ("fp8 attention drops the V scale", "(e4m3_value(v8[kv + (size_t)n * d + i]) * v_scale[g])",
     "(e4m3_value(v8[kv + (size_t)n * d + i]))"),
    ("projection reads the weight transposed", "load_value(p, ((size_t)h * A + a) * d + j, dtype)",
     "load_value(p, ((size_t)h * d + j) * A + a, dtype)"),
    ("K projected with the query weights", "project_heads(x, pk, k,", "project_heads(x, pq, k,"),
    ("projection drops the last input feature", "for (int a = 0; a < A; ++a)\n                s += load_value(x,",
     "for (int a = 0; a < A - 1; ++a)\n                s += load_value(x,"),
    ("q read reversed", "load_value(q, q_off + i, dtype)", "load_value(q, q_off + (d - 1 - i), dtype)"),
    ("wrong sign of logits", "w[n] = dot * scale;", "w[n] = -dot * scale;"),
    ("meanpool sums instead of averaging", "w_out[(size_t)g * per_head + e] = s / n_rep;",
     "w_out[(size_t)g * per_head + e] = s;"),
    ("append does not advance the length", "seq_lens[b] = L + 1;", "seq_lens[b] = L;"),
    ("append writes the wrong row", "* Nmax + (size_t)L) * row;", "* Nmax + (size_t)L + 1) * row;"),
]


def _failures():
    failed = []
    for pin in PIN_BATTERY:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(getattr(pin, "__name__", "lambda"))
    return failed


def test_every_pin_passes_on_the_real_oracle():
    assert _failures() == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", str(so), str(mutant), "-lm"])
    with oracle.use_library(str(so)):
        failed = _failures()
    assert failed, f"no pin caught the planted mistake: {name}"
