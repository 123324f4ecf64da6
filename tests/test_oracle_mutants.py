"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one mistake in a copy of oracle/mp_oracle.c — a swapped
operand, a dropped term, a wrong sign, exponent, comparison or index —
compiles it, swaps it in for the real oracle and runs the pins of
test_oracle_pins.py until one fails. Every mutant must be caught; the
unmodified oracle must pass them all.

The hash is mutated only where a mistake leaves a worse mixer (a dropped
multiply or xor-shift round), which the avalanche pin catches. Its constants
and shift amounts, and changes that leave an equally good mixer (the seed
xored instead of added, a shift reversed), are not: the pages print no test
vector for SquirrelNoise5, so those are pinned only through the statistical
checks, which a different but equally good mixer would pass.
"""
import os
import subprocess

import pytest

import oracle
from oracle import build as oracle_build
import test_oracle_pins as P
from conftest import read_golden

SRC = oracle_build.SRC
HDR = oracle_build.HDR

MUTANTS = {
    "lerp operands swapped":
        ("return fmaf(w, end, fmaf(-w, start, start));", "return fmaf(w, start, fmaf(-w, end, end));"),
    "eps inside the square root":
        ("const float denom = sqrtf(v_hat) + eps;", "const float denom = sqrtf(v_hat + eps);"),
    "decay with the wrong sign":
        ("const float update = m_hat / denom + wd * old;", "const float update = m_hat / denom - wd * old;"),
    "update with the wrong sign":
        ("const float p = old - lr * update;", "const float p = old + lr * update;"),
    "bias correction at t - 1":
        ("*bc1 = (float)(1.0 - pow((double)beta1, (double)t));",
         "*bc1 = (float)(1.0 - pow((double)beta1, (double)(t - 1)));"),
    "second moment not bias-corrected":
        ("const float v_hat = v_new / bc2;", "const float v_hat = v_new;"),
    "bias corrections swapped":
        ("const float m_hat = m_new / bc1;", "const float m_hat = m_new / bc2;"),
    "beta1 used for the second moment":
        ("const float v_new = lerp_two_fma(gg, v[i], beta2);", "const float v_new = lerp_two_fma(gg, v[i], beta1);"),
    "grad scale dropped":
        ("const float grad = scale * bf16_bits_to_float(grads[i]);",
         "const float grad = bf16_bits_to_float(grads[i]);"),
    "decay on every tensor":
        ("const float wd = table[k].decay ? weight_decay : 0.0f;", "const float wd = weight_decay;"),
    "decay on the 1D tensors instead":
        ("const float wd = table[k].decay ? weight_decay : 0.0f;",
         "const float wd = table[k].decay ? 0.0f : weight_decay;"),
    "master keeps the old weight":
        ("        master[i] = p;", "        master[i] = old;"),
    "draw keyed on the local index":
        ("params[i] = oracle_sr(p, gi, seed);", "params[i] = oracle_sr(p, i, seed);"),
    "rounding compares with >=":
        ("if (lo16 > rand16)", "if (lo16 >= rand16)"),
    "rounding always truncates":
        ("return (uint16_t)(truncated + 1u);", "return (uint16_t)truncated;"),
    "NaN not made canonical":
        ("    if (isnan(x))\n        return 0x7FC0u;", "    if (0)\n        return 0x7FC0u;"),
    "norm sums |g| instead of g^2":
        ("        s += g * g;", "        s += g < 0 ? -g : g;"),
    "norm without the square root":
        ("const float nf = (float)sqrt(s);", "const float nf = (float)s;"),
    "clip rule inverted":
        ("return q < 1.0f ? q : 1.0f;", "return q > 1.0f ? q : 1.0f;"),
    "outlier: sample instead of population std":
        ("const double sd = sqrt(ss / ORACLE_OUTLIER_WINDOW);",
         "const double sd = sqrt(ss / (ORACLE_OUTLIER_WINDOW - 1));"),
    "outlier: z with the wrong sign":
        ("zz = (x - mean) / sd;", "zz = (mean - x) / sd;"),
    "fp16: rounds up on a tie with the draw":
        ("const uint32_t up = frac16 > rand16 ? 1u : 0u;", "const uint32_t up = frac16 >= rand16 ? 1u : 0u;"),
    "fp16: wrong step past the largest finite value":
        ("lo == 0x7BFF ? 32.0 :", "lo == 0x7BFF ? 16.0 :"),
    "fp16: NaN not made canonical":
        ("    if (isnan(x))\n        return 0x7E00u;", "    if (0)\n        return 0x7E00u;"),
    "accumulate: contribution dropped":
        ("const float sum = bf16_bits_to_float(acc[i]) + delta[i];",
         "const float sum = bf16_bits_to_float(acc[i]);"),
    "accumulate: draw keyed on the local index":
        ("acc[i] = oracle_sr(sum, global_offset + i, seed);", "acc[i] = oracle_sr(sum, i, seed);"),
    "norm pieces: running total ignored":
        ("double oracle_sumsq_from(double s, const uint16_t* grads, uint64_t n)\n{\n",
         "double oracle_sumsq_from(double s, const uint16_t* grads, uint64_t n)\n{\n    s = 0.0;\n"),
    "ZeRO-1 norm: parts added in reverse rank order":
        ("    for (int32_t r = 0; r < count; ++r)\n        s += parts[r];",
         "    for (int32_t r = count - 1; r >= 0; --r)\n        s += parts[r];"),
    "ZeRO-1 norm: last part dropped":
        ("    for (int32_t r = 0; r < count; ++r)\n        s += parts[r];",
         "    for (int32_t r = 0; r + 1 < count; ++r)\n        s += parts[r];"),
    "ZeRO-1 norm without the square root":
        ("const float root = (float)sqrt(s);", "const float root = (float)s;"),
    "lr: warm-up one step late":
        ("return (float)(hi * (double)t / (double)warmup);", "return (float)(hi * (double)(t - 1) / (double)warmup);"),
    "lr: cosine upside down":
        ("lr = lo + (hi - lo) * (1.0 + cos(pi * p)) / 2.0;", "lr = lo + (hi - lo) * (1.0 - cos(pi * p)) / 2.0;"),
    "lr: progress not clamped":
        ("    if (p > 1.0)\n        p = 1.0;", "    if (p > 2.0)\n        p = 1.0;"),
    "lr: WSD decays from the start of its last fraction's complement":
        ("lr = (p <= 1.0 - f) ? hi : hi - (hi - lo) * (p - (1.0 - f)) / f;",
         "lr = (p <= f) ? hi : hi - (hi - lo) * (p - f) / (1.0 - f);"),
    "lr: linear decays to zero":
        ("lr = hi - (hi - lo) * p;", "lr = hi - hi * p;"),
    "hash: final xor-shift dropped":
        ("    bits ^= bits >> 17;\n", ""),
    "hash: a middle multiply dropped":
        ("    bits *= 0x6C736F4Bu;\n", ""),
    "hash: last multiply dropped":
        ("    bits *= 0x1B56C4F5u;\n", ""),
    "outlier: non-finite norms enter the window":
        ("    if (isfinite(x)) {\n        st->window", "    if (1) {\n        st->window"),
}


def _pins():
    """The pins, cheapest first, as zero-argument callables."""
    g = read_golden
    return [
        ("bias multipliers", lambda: P.test_bias_correction_multipliers_match_printed_values(g)),
        ("bias 1 - beta^t", P.test_bias_correction_is_one_minus_beta_to_the_t),
        ("clip rule", P.test_clip_scale_rule),
        ("norm of ones", P.test_norm_of_all_ones_is_sqrt_n),
        ("norm of powers of two", P.test_norm_of_power_of_two_pattern_is_exact),
        ("norm vs fsum", P.test_norm_matches_math_fsum),
        ("norm non-finite", P.test_norm_with_nonfinite_grads_gives_nan_scale),
        ("sr specials", P.test_sr_special_values),
        ("sr representable", P.test_sr_leaves_bf16_representable_values_unchanged),
        ("first step a", lambda: P.test_first_step_closed_form(1e-3, 0.1, 1e-8)),
        ("first step b", lambda: P.test_first_step_closed_form(0.1, 0.5, 1e-8)),
        ("first step c", lambda: P.test_first_step_closed_form(0.05, 0.0, 1e-3)),
        ("lr sign(g)", P.test_first_step_moves_each_weight_by_lr_sign_g_when_eps_is_tiny),
        ("no master", P.test_no_master_variant_reads_old_weight_from_bf16),
        ("non-finite scale", P.test_nonfinite_scale_writes_nothing),
        ("decay only 2D", P.test_zero_gradient_leaves_1d_tensors_unchanged_and_decays_2d),
        ("sr exhaustive", lambda: P.test_sr_exhaustive_over_all_draws(P.SR_VALUES[0])),
        ("sr half-way", lambda: P.test_sr_halfway_values_from_bf16_facts(g)),
        ("outlier vs pstdev", P.test_outlier_zscore_matches_statistics_pstdev),
        ("outlier closed form", P.test_outlier_closed_form_and_skip),
        ("outlier window", P.test_outlier_window_ignores_nonfinite_norms_and_slides),
        ("resume", P.test_resume_rebuilds_bf16_bit_identically),
        ("shards", lambda: P.test_sharded_steps_equal_whole_buffer_steps(True)),
        ("torch AdamW fp64", P.test_sixteen_steps_track_torch_adamw_fp64),
        ("sr tracks small updates", P.test_sr_tracks_small_updates_where_round_to_nearest_stalls),
        ("fp16 keeps fp16", P.test_sr_fp16_keeps_every_fp16_value),
        ("fp16 exhaustive", lambda: P.test_sr_fp16_exhaustive_over_draws(1.0 + 2 ** -12)),
        ("fp16 exhaustive near max", lambda: P.test_sr_fp16_exhaustive_over_draws(65504.5)),
        ("fp16 half-way", lambda: P.test_sr_fp16_halfway_value_from_the_pages(g)),
        ("fp16 specials", P.test_sr_fp16_special_values_and_unbiasedness),
        ("accumulate zero", P.test_accumulate_sr_adding_zero_changes_nothing),
        ("accumulate exact", P.test_accumulate_sr_exact_when_the_sum_is_representable),
        ("accumulate unbiased", P.test_accumulate_sr_is_unbiased_over_seeds),
        ("accumulate shards", P.test_accumulate_sr_keeps_small_contributions_and_shards),
        ("norm in pieces", P.test_sumsq_continued_in_pieces_equals_one_pass),
        ("ZeRO-1 norm exact", P.test_norm_from_parts_equals_whole_buffer_norm_on_exact_sums),
        ("ZeRO-1 norm order", P.test_norm_from_parts_adds_in_rank_order_in_fp64),
        ("ZeRO-1 norm bound", P.test_norm_from_parts_within_rounding_of_the_exact_sum),
        ("lr warm-up", lambda: [P.test_lr_warmup_is_linear_and_reaches_the_peak(k) for k in range(4)]),
        ("lr constant", P.test_lr_constant_after_warmup),
        ("lr cosine", P.test_lr_cosine_closed_forms),
        ("lr linear", P.test_lr_linear_closed_forms),
        ("lr WSD", P.test_lr_wsd_closed_forms),
        ("lr invalid", P.test_lr_rejects_invalid_arguments),
        ("noise avalanche", P.test_noise_avalanche),
    ]


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    d = tmp_path / "mutant"
    d.mkdir()
    (d / "mp_oracle.c").write_text(src.replace(old, new))
    (d / "mp_oracle.h").write_text(open(HDR).read())
    lib = d / "mutant.so"
    flags = [f for f in oracle_build.CFLAGS if f != "-Werror"]
    subprocess.run(["gcc", *flags, str(d / "mp_oracle.c"), "-o", str(lib), "-lm"], check=True)
    return oracle.load_library(str(lib))


def _first_failing_pin(lib):
    saved = oracle._lib
    oracle._lib = lib
    try:
        for name, pin in _pins():
            try:
                pin()
            except AssertionError:
                return name
        return None
    finally:
        oracle._lib = saved


def test_unmodified_oracle_passes_every_pin():
    assert _first_failing_pin(oracle.lib()) is None


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_every_planted_mistake_is_caught(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    lib = _build_mutant(tmp_path, old, new)
    caught_by = _first_failing_pin(lib)
    assert caught_by is not None, f"no pin catches: {mutant}"
