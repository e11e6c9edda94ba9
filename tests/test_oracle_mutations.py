"""Mutation check of the oracle's pins.

Each entry below is a plausible mistake in the oracle (a swapped operand, a
wrong sign or index, a dropped term, a misread format field).  The test plants
it in a copy of the C oracle source, builds that copy, points the oracle
wrapper at it, and requires at least one pin of test_oracle_pins.py to fail:
a pin set that passes a broken oracle does not pin it.  The unaltered copy,
built the same way, must pass every pin.  Nothing here touches the product or
the oracle's own source.
"""
from __future__ import annotations

import os

import pytest

import oracle
from oracle import build as oracle_build
from tests import test_oracle_pins as pins

# (text in oracle/flint_moe_ref.c, what the mistake puts there instead)
MUTATIONS = {
    "gate and up swapped": (
        "act[i] = g / (1.0 + exp(-g)) * u;", "act[i] = u / (1.0 + exp(-u)) * g;"),
    "SiLU sign flipped": (
        "act[i] = g / (1.0 + exp(-g)) * u;", "act[i] = g / (1.0 + exp(g)) * u;"),
    "tie goes to the higher index": (
        "logits[e] > logits[best]", "logits[e] >= logits[best]"),
    "sigmoid sign flipped": (
        "w[j] = 1.0 / (1.0 + exp(-score_in));", "w[j] = 1.0 / (1.0 + exp(score_in));"),
    "weights not renormalised": (
        "for (int j = 0; j < k; ++j) w[j] /= ssum;", "for (int j = 0; j < k; ++j) w[j] /= 1.0;"),
    "logit offsets ignored": (
        "logits[e] = acc + (bias ? (double)bias[e] : 0.0);", "logits[e] = acc;"),
    "select-only weights take the offsets": (
        "d->offset_mode == 1 ? raw[best] : logits[best]", "logits[best]"),
    "select-only offsets ignored in the ranking": (
        "logits[e] = acc + (bias ? (double)bias[e] : 0.0);",
        "logits[e] = acc + (bias && d->offset_mode != 1 ? (double)bias[e] : 0.0);"),
    "shared expert dropped": (
        "for (int h = 0; h < H; ++h) o[h] += y[h];",
        "for (int h = 0; h < H; ++h) o[h] += 0.0 * y[h];"),
    "routing weight ignored": (
        "o[h] += w[(size_t)t * k + j] * y[h];", "o[h] += y[h];"),
    "residual dropped": (
        "o[h] = bf16_value(residual[(size_t)t * H + h]);", "o[h] = 0.0;"),
    "down projection rows shifted by one": (
        "acc += mat_at(m2, r, i) * act[i];", "acc += mat_at(m2, (r + 1) % H, i) * act[i];"),
    "e2m1 nibbles swapped": (
        "(k & 1) ? (byte >> 4) : (byte & 15)", "(k & 1) ? (byte & 15) : (byte >> 4)"),
    "e2m1 subnormal misread": ("exp == 0 ? 0.5 * man", "exp == 0 ? 1.0 * man"),
    "e4m3 exponent bias off by one": (
        "mag = ldexp(1.0 + man / 8.0, exp - 7);", "mag = ldexp(1.0 + man / 8.0, exp - 8);"),
    "gate / up tensor scales swapped": (
        "m13->ts_lo = ts13[0];\n    m13->ts_hi = ts13[1];",
        "m13->ts_lo = ts13[1];\n    m13->ts_hi = ts13[0];"),
    "RoPE rotation sign flipped": ("out[i] = lo * c - hi * s;", "out[i] = lo * c + hi * s;"),
    "RoPE frequency exponent halved": (
        "pow(theta, -2.0 * i / D)", "pow(theta, -1.0 * i / D)"),
    "RoPE position ignored": ("double a = (double)pos * pow(", "double a = pow("),
    "RoPE pairs element i with i + 1": (
        "double lo = out[i], hi = out[i + half];\n      out[i] = lo * c - hi * s;\n      out[i + half] = hi * c + lo * s;",
        "double lo = out[2 * i], hi = out[2 * i + 1];\n      out[2 * i] = lo * c - hi * s;\n      out[2 * i + 1] = hi * c + lo * s;"),
    "Q/K norm gain ignored": (
        "out[i] = bf16_value(x[i]) * inv * bf16_value(g[i]);", "out[i] = bf16_value(x[i]) * inv;"),
    "Q/K norm eps dropped": ("double inv = 1.0 / sqrt(ss / D + eps);", "double inv = 1.0 / sqrt(ss / D);"),
    "query heads take the key gain": (
        "qk_head(D, x + (size_t)h * D, q_norm,", "qk_head(D, x + (size_t)h * D, k_norm,"),
    "value heads read from the key heads": (
        "bf16_value(x[(size_t)(nq + nkv + h) * D + i]);", "bf16_value(x[(size_t)(nq + h) * D + i]);"),
}

# The pins run against each build: all of test_oracle_pins.py's CPU-quick pins.
PINS = [
    ("brute force, tiny, batch 8 with offsets", lambda: pins.test_matches_dense_brute_force_tiny(3, 8, True, False)),
    ("brute force, tiny, batch 17", lambda: pins.test_matches_dense_brute_force_tiny(4, 17, False, False)),
    ("brute force, tiny, batch 8, offsets for selection only",
     lambda: pins.test_matches_dense_brute_force_tiny(6, 8, True, True)),
    ("x = 0 with offsets for selection only",
     pins.test_zero_input_select_only_offsets_rank_and_weights_are_equal),
    ("first k of a full sort, weights sum to 1",
     pins.test_selection_is_first_k_of_full_sort_and_weights_sum_to_one),
    ("token permutation", pins.test_token_permutation_permutes_outputs_exactly),
    ("batch invariance", pins.test_batch_invariance_row_alone_equals_row_in_batch),
    ("x = 0", pins.test_zero_input_gives_lowest_indices_equal_weights_and_residual),
    ("x = 0 with offsets", pins.test_zero_input_with_offsets_ranks_by_offsets),
    ("crafted router, identity-embedded experts",
     pins.test_crafted_router_and_identity_embedded_experts_closed_form),
    ("identical experts", pins.test_identical_experts_reduce_to_one_expert),
    ("SiLU expression", pins.test_silu_form_matches_page_expression),
    ("e2m1 codes", pins.test_e2m1_all_codes_match_spec_table),
    ("e4m3 codes", pins.test_e4m3_all_codes_match_library_decode_and_spec_points),
    ("NVFP4 = BF16 on dequantised weights", pins.test_nvfp4_layer_equals_bf16_layer_on_dequantised_weights),
    ("Q/K norm + RoPE, hand-computed head", pins.test_qk_norm_rope_hand_computed_head),
    ("Q/K norm eps under the root", pins.test_qk_norm_eps_sits_under_the_root),
    ("Q/K norm + RoPE invariants", pins.test_qk_norm_rope_invariants),
    ("RoPE relative position", pins.test_rope_scores_depend_on_relative_position_only),
]


def _failing_pins(first_only=False):
    failed = []
    for name, pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(name)
            if first_only:
                break
    return failed


def _build_variant(tmp_path, tag, text):
    src = tmp_path / ("ref_%s.c" % tag)
    src.write_text(text)
    return oracle.load(oracle_build.compile_to(str(src), str(tmp_path / ("ref_%s.so" % tag))))


@pytest.fixture(scope="module")
def source():
    with open(oracle_build.SRC) as f:
        return f.read()


def test_unaltered_copy_passes_every_pin(tmp_path, monkeypatch, source):
    monkeypatch.setattr(oracle, "_lib", _build_variant(tmp_path, "orig", source))
    assert _failing_pins() == []


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_each_planted_mistake_fails_a_pin(tmp_path, monkeypatch, source, mutation):
    old, new = MUTATIONS[mutation]
    assert source.count(old) == 1, "mutation site not found once: %r" % old
    tag = "m%d" % sorted(MUTATIONS).index(mutation)
    monkeypatch.setattr(oracle, "_lib", _build_variant(tmp_path, tag, source.replace(old, new)))
    assert _failing_pins(first_only=True), "no pin caught: %s" % mutation
    assert os.path.exists(oracle_build.SRC)
