"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is the committed C source with one textual change, compiled on
the CPU into a temporary library; the committed oracle is never touched.
"""
import os
import subprocess

import pytest

import oracle
from oracle import build as oracle_build
import oracle_pins

MUTANTS = {
    "sign_flip_in_sum": ("acc = acc + oracle_bf16_to_f32(partials[k][idx]);",
                         "acc = acc - oracle_bf16_to_f32(partials[k][idx]);"),
    "dropped_last_rank": ("for (int k = 1; k < n; ++k)",
                          "for (int k = 1; k < n - 1; ++k)"),
    "reverse_rank_order": ("acc = acc + oracle_bf16_to_f32(partials[k][idx]);",
                           "acc = acc + oracle_bf16_to_f32(partials[n - k][idx]);"),
    "fp64_accumulator": ("float acc = oracle_bf16_to_f32(partials[0][idx]);",
                         "double acc = oracle_bf16_to_f32(partials[0][idx]);"),
    "no_two_stage_rounding": ("if (two_stage)\n        acc =", "if (0)\n        acc ="),
    "residual_dropped": ("float r = acc + oracle_bf16_to_f32(residual[base + j]);",
                         "float r = acc;"),
    "eps_outside_sqrt": ("1.0 / sqrt(ss / (double)H + eps)", "1.0 / (sqrt(ss / (double)H) + eps)"),
    "mean_over_ranks": ("ss / (double)H + eps", "ss / (double)n + eps"),
    "weight_reversed": ("oracle_bf16_to_f32(weight[j])", "oracle_bf16_to_f32(weight[H - 1 - j])"),
    "row_stride_wrong": ("const int64_t base = i * H;", "const int64_t base = i * (H - 1);"),
    "truncating_round": ("nearbyint(ldexp(ax, -qexp))", "trunc(ldexp(ax, -qexp))"),
    "ties_away": ("nearbyint(ldexp(ax, -qexp))", "round(ldexp(ax, -qexp))"),
    "one_stage_also_rounds": ("if (two_stage)\n        acc =", "if (1)\n        acc ="),
    "first_rank_dropped": ("float acc = oracle_bf16_to_f32(partials[0][idx]);",
                           "float acc = 0.0f;"),
    "eps_dropped": ("1.0 / sqrt(ss / (double)H + eps)", "1.0 / sqrt(ss / (double)H)"),
    "square_sum_of_rounded_residual": (
        "ss += (double)r * (double)r;",
        "{ double q = oracle_bf16_to_f32(residual_out[base + j]); ss += q * q; }"),
    "output_from_rounded_residual": (
        "double y = (double)r_scratch[j] * inv",
        "double y = (double)oracle_bf16_to_f32(residual_out[base + j]) * inv"),
    "weight_ignored": ("* (double)oracle_bf16_to_f32(weight[j]);", "* 1.0;"),
    "mean_over_h_minus_one": ("ss / (double)H + eps", "ss / (double)(H - 1) + eps"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle_build.SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle_build.CFLAGS, "-w", "-o", str(so), str(c), "-lm", "-lpthread"],
                   check=True)
    fails = oracle_pins.run_all(oracle.Oracle(str(so)))
    assert fails, f"planted mistake {name!r} passed every pin"
