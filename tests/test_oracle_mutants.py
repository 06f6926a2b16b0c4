"""Planted mistakes: each test compiles a copy of the oracle with one plausible
slip (on the CPU, in a temporary directory) and checks that the pins in
test_oracle_pins.py reject it.  The committed oracle is never altered."""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "gqa_map_modulo": ("const int g = (int)(((long)h * H_kv) / H_q);\n    contig_ctx c;",
                       "const int g = h % H_kv;\n    contig_ctx c;"),
    "scale_dropped": ("scores[j] = dot * scale;", "scores[j] = dot;"),
    "causal_off_by_one": ("const int n = causal ? i + 1 : S;", "const int n = causal ? i : S;"),
    "value_from_key_rows": ("const uint16_t *v = val(ctx, j);", "const uint16_t *v = key(ctx, j);"),
    "page_slot_swapped": ("* x->bs + (t % x->bs)) * (long)x->D;", "* x->bs + (t / x->bs) % x->bs) * (long)x->D;"),
    "lse_missing_max": ("*lse = M + log(sum);", "*lse = log(sum);"),
    "combine_weight_by_max": ("const double w = exp(lp[i] - L);", "const double w = exp(lp[i] - M);"),
    "decode_gqa_map": ("c.g = (int)(((long)h * H_kv) / H_q);\n    attend_one(q + ((long)n * H_q + h) * D",
                       "c.g = (int)(h % H_kv);\n    attend_one(q + ((long)n * H_q + h) * D"),
    "paged_prefill_no_prefix_offset": ("const int n = causal ? Lkv - Lq + i + 1 : Lkv;",
                                       "const int n = causal ? i + 1 : Lkv;"),
    "rope_sin_sign": ("o[i] = y[i] * c - y[i + half] * s;", "o[i] = y[i] * c + y[i + half] * s;"),
    "rope_frequency_exponent": ("pow(base, -2.0 * i / D)", "pow(base, -1.0 * i / D)"),
    "rope_position_by_row": ("const int t = (int)(r / H);", "const int t = (int)(r % T);"),
    "norm_eps_dropped": ("sqrt(ss / D + eps)", "sqrt(ss / D)"),
    "norm_mean_over_half": ("sqrt(ss / D + eps)", "sqrt(ss / half + eps)"),
    "norm_weight_dropped": ("y[d] = oracle_half_to_double(w[d]) * y[d] / rms;", "y[d] = y[d] / rms;"),
}

PINS = [
    lambda: [pins.test_prefill_matches_torch_sdpa_float64(s, c) for s in pins.SHAPES for c in (True, False)],
    pins.test_prefill_gqa_map_distinguishes_groups,
    lambda: pins.test_identical_k_rows_give_mean_of_allowed_v(True),
    pins.test_causal_row0_is_v0_and_zero_keys_lse,
    lambda: pins.test_decode_paged_equals_last_prefill_row(5),
    pins.test_decode_matches_sdpa_on_gathered_keys_ragged,
    lambda: pins.test_lse_merge_of_segments_equals_whole([0, 1, 2, 33, 40]),
    pins.test_lse_merge_two_known_partials,
    pins.test_prefill_paged_equals_last_rows_of_full_causal_prefill,
    lambda: pins.test_rope_frequencies_are_geometric_from_one(128),
    pins.test_rope_equals_complex_rotation,
    lambda: [pins.test_qk_norm_equals_torch_rms_norm_at_position_zero(s) for s in (1.0, 1e-4)],
    pins.test_qk_norm_then_rope_order_and_weights,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(src), "-lm"],
                   check=True)
    failures = 0
    with oracle.variant(str(lib)):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failures += 1
    assert failures >= 1, f"no pin caught the planted mistake {name}"
