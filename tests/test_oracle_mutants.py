"""Plant one plausible mistake at a time in a copy of the oracle source (on the
CPU) and check that the pins catch every one of them.  The shipped oracle is
untouched; each mutant is compiled into a temporary directory."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import test_oracle as pins
from tests import test_oracle_mhc as mhc_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ar_oracle.c")

# (name, original text, mutated text): each is one small, plausible slip.
MUTANTS = [
    ("drop shared term", "y_r += s;", "(void)s;"),
    ("shared added for rank 0 only", "if (S) {\n                double s", "if (S && r == 0) {\n                double s"),
    ("residual subtracted", "h_row[j] = y + res;", "h_row[j] = y - res;"),
    ("residual dropped", "h_row[j] = y + res;", "h_row[j] = y;"),
    ("perm slots reversed against the weights", "int64_t row = perm[t * K + k];", "int64_t row = perm[t * K + (K - 1 - k)];"),
    ("perm ignored (identity gather)", "int64_t row = perm[t * K + k];", "int64_t row = t * K + k;"),
    ("weights of token 0 for every token", "(double)w[t * K + k]", "(double)w[k]"),
    ("weights ignored", "(double)w[t * K + k] *", "1.0 *"),
    ("rank 0 buffer for every rank", "bf16_bits_to_double(E[r][row * H + j])", "bf16_bits_to_double(E[0][row * H + j])"),
    ("weight_bias dropped", "bf16_bits_to_double(gamma[j]) + weight_bias", "bf16_bits_to_double(gamma[j])"),
    ("gamma dropped", "bf16_bits_to_double(gamma[j]) + weight_bias", "1.0 + weight_bias"),
    ("eps outside the sqrt", "sqrt(ms + eps)", "(sqrt(ms) + eps)"),
    ("sum of squares, not mean", "double ms = ssq / (double)H;", "double ms = ssq;"),
    ("rms instead of inverse rms", "out_row[j] = hj / denom * g;", "out_row[j] = hj * denom * g;"),
    ("bf16 decoded one bit short", "((uint32_t)b) << 16", "((uint32_t)b) << 15"),
    ("last column of the norm skipped", "for (int j = 0; j < H; ++j) {\n        double hj = h_bf16 ? oracle_round_bf16(h_row[j]) : h_row[j];\n        ssq",
     "for (int j = 0; j + 1 < H; ++j) {\n        double hj = h_bf16 ? oracle_round_bf16(h_row[j]) : h_row[j];\n        ssq"),
    ("rounding quantum off by one", "int q = e - 8;", "int q = e - 9;"),
    ("shared gate dropped", "double s = g * bf16_bits_to_double(S[r][t * H + j]);",
     "double s = bf16_bits_to_double(S[r][t * H + j]);"),
    ("shared gate sign flipped", "1.0 / (1.0 + exp(-(double)gate[t]))", "1.0 / (1.0 + exp((double)gate[t]))"),
    ("hc_post mix matrix transposed", "comb[(t * hc + i) * hc + k]", "comb[(t * hc + k) * hc + i]"),
    ("hc_post reduced output dropped", "double o = (double)post[t * hc + i] * y;", "double o = 0.0;"),
    ("hc_post post weight of stream 0 for all", "double o = (double)post[t * hc + i] * y;",
     "double o = (double)post[t * hc] * y;"),
    ("hc_post all-reduce over rank 0 only", "for (int r = 0; r < R; ++r)\n                y += bf16_bits_to_double(partials",
     "for (int r = 0; r < 1; ++r)\n                y += bf16_bits_to_double(partials"),
    ("hc_post streams of token 0", "bf16_bits_to_double(x[(t * hc + k) * H + j])", "bf16_bits_to_double(x[(0 * hc + k) * H + j])"),
]

PINS = [
    lambda: [pins.test_brute_force_2x4(R, K, sh, d) for R in (1, 2) for K in (0, 1, 2)
             for sh in (True, False) for d in (False, True) if K or sh],
    pins.test_brute_force_tiny_config,
    lambda: pins.test_perm_decode_exact(8, 8, 64, 16),
    pins.test_reduces_to_plain_rms_norm,
    pins.test_gemma_weight_bias_equivalence,
    pins.test_shared_partial_counted_once_per_rank,
    pins.test_round_bf16_matches_fp32_to_bf16_for_fp32_values,
    lambda: [pins.test_gated_brute_force_2x4(R, K) for R, K in ((1, 1), (2, 2), (2, 0))],
    pins.test_gate_scales_only_the_shared_term,
    lambda: [mhc_pins.test_mhc_brute_force(R, hc) for R, hc in ((1, 1), (2, 2), (2, 4), (3, 4))],
    mhc_pins.test_mhc_identity_mix_returns_the_streams,
    mhc_pins.test_mhc_pure_all_reduce_matches_the_main_oracle,
    mhc_pins.test_mhc_single_stream_is_the_residual_add,
    mhc_pins.test_mhc_stream_relabelling,
    mhc_pins.test_mhc_hand_example,
]


def _caught() -> list:
    hits = []
    for i, pin in enumerate(PINS):
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, IndexError, ValueError):
            hits.append(i)
    return hits


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.GCC_FLAGS, "-o", str(so), str(mut), "-lm"], check=True)
    with oracle._swap_library(str(so)):
        hits = _caught()
    assert hits, f"no pin caught the planted mistake '{name}'"


def test_unmutated_copy_passes_every_pin(tmp_path):
    so = tmp_path / "libcopy.so"
    subprocess.run(["gcc", *oracle.GCC_FLAGS, "-o", str(so), SRC, "-lm"], check=True)
    with oracle._swap_library(str(so)):
        assert _caught() == []
