"""Plants plausible mistakes in a copy of the oracle's C source (on the CPU)
and checks that the pins reject every one: a pin that a dropped term, a wrong
sign, a swapped index or a reversed tie rule would pass is no pin."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_nvfp4 as nv
from tests import test_oracle_pins as pins
from tests import test_oracle_router_awq as ra
from w4a16_group_quantized_moe_gb300 import inputs

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

# (name, original text, mutated text); each original must occur exactly once
MUTANTS = [
    ("nibble order reversed", "(qweight[qword] >> (4 * (kk % 8)))",
     "(qweight[qword] >> (4 * (7 - kk % 8)))"),
    ("zero nibble taken by column", "(qzeros[zword] >> (4 * (n % 8)))",
     "(qzeros[zword] >> (4 * (kk % 8)))"),
    ("zero point sign flipped", "return (double)(q - z) * s;", "return (double)(q + z) * s;"),
    ("scale of group 0 everywhere", "scales[((size_t)e * N + n) * G + kk / 32]",
     "scales[((size_t)e * N + n) * G]"),
    ("gate used for up", "u += xv * oracle_dequant(w13q, w13s, w13z, 2 * I, H, e, I + i, kk);",
     "u += xv * oracle_dequant(w13q, w13s, w13z, 2 * I, H, e, i, kk);"),
    ("silu dropped", "hrow[i] = silu(g) * u;", "hrow[i] = g * u;"),
    ("silu sign", "return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    ("no renormalisation", "topk_w[(size_t)t * k + j] = prob[e] / selected_mass;",
     "topk_w[(size_t)t * k + j] = prob[e];"),
    ("tie goes to higher index", "return a < b;", "return a > b;"),
    ("combine weight dropped", "acc += topk_w[(size_t)t * k + j] * y[(size_t)r * H + n];",
     "acc += y[(size_t)r * H + n];"),
    ("segment order reversed", "for (int p = 0; p < P; ++p)\n            if (topk_ids[p] == e)",
     "for (int p = P - 1; p >= 0; --p)\n            if (topk_ids[p] == e)"),
    ("last group of K dropped", "for (int kk = 0; kk < H; ++kk) {",
     "for (int kk = 0; kk < H - 32; ++kk) {"),
]

# planted mistakes in the NVFP4 functions, checked by the NVFP4 pins
NVFP4_MUTANTS = [
    ("e2m1 sign dropped", "return sign ? -v : v;\n}\n\n/* FP8 E4M3", "return v;\n}\n\n/* FP8 E4M3"),
    ("e2m1 subnormal as normal", "double v = expo == 0 ? 0.5 * mant : ldexp(1.0 + 0.5 * mant, expo - 1);",
     "double v = ldexp(1.0 + 0.5 * mant, expo - 1);"),
    ("e4m3 bias off by one", "v = ldexp(1.0 + (double)mant / 8.0, expo - 7);",
     "v = ldexp(1.0 + (double)mant / 8.0, expo - 8);"),
    ("block of 32 instead of 16", "bscale[((size_t)e * N + n) * (K / 16) + kk / 16]",
     "bscale[((size_t)e * N + n) * (K / 16) + kk / 32]"),
    ("per-expert scale dropped", "return oracle_e2m1_to_double(nib) * bs * (double)gscale[e];",
     "return oracle_e2m1_to_double(nib) * bs;"),
    ("nvfp4 gate used for up", "u += xv * oracle_dequant_nvfp4(c13, b13, g13, 2 * I, H, e, I + i, c);",
     "u += xv * oracle_dequant_nvfp4(c13, b13, g13, 2 * I, H, e, i, c);"),
    ("nvfp4 silu dropped", "hrow[i] = u * silu(g);", "hrow[i] = u * g;"),
]

CHECKS = [
    pins.test_dequant_unpacks_hand_derived_words,
    pins.test_route_hand_derived_cases,
    lambda m: pins.test_route_matches_brute_force_sort(m, 7, 512, 10),
    lambda m: pins.test_align_matches_bincount_cumsum_and_stable_sort(m, 300, 64, 6),
    lambda m: pins.test_layer_matches_dense_brute_force(m, pins.SHAPES[0]),
    lambda m: pins.test_layer_matches_dense_brute_force(m, pins.SHAPES[1]),
    pins.test_layer_constant_closed_form,
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, orig, mut):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for '{name}' not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(orig, mut))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fvisibility=hidden", str(mpath), "-o", str(lib), "-lm"])
    caught = []
    with oracle.using_library(str(lib)):
        for check in CHECKS:
            try:
                check(oracle)
            except AssertionError:
                caught.append(check)
    assert caught, f"no pin rejects the planted mistake '{name}'"


NVFP4_CHECKS = [
    nv.test_e2m1_matches_the_specification_table,
    nv.test_e4m3_matches_torch_for_every_byte,
    nv.test_dequant_hand_derived_word,
    nv.test_dequant_uses_the_block_of_sixteen,
    lambda m: nv.test_layer_matches_dense_brute_force(m, nv.SHAPES[0]),
    nv.test_layer_constant_closed_form,
]


@pytest.mark.parametrize("name,orig,mut", NVFP4_MUTANTS, ids=[m[0] for m in NVFP4_MUTANTS])
def test_planted_nvfp4_mistake_is_caught(tmp_path, name, orig, mut):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for '{name}' not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(orig, mut))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fvisibility=hidden", str(mpath), "-o", str(lib), "-lm"])
    caught = []
    with oracle.using_library(str(lib)):
        for check in NVFP4_CHECKS:
            try:
                check(oracle)
            except AssertionError:
                caught.append(check)
    assert caught, f"no pin rejects the planted mistake '{name}'"


# planted mistakes in the router-logits product and the AWQ import
RA_MUTANTS = [
    ("router matrix read transposed", "oracle_half_to_double(wr[(size_t)e * H + c]);",
     "oracle_half_to_double(wr[(size_t)c * E + e]);"),
    ("router last term dropped", "for (int c = 0; c < H; ++c)\n                acc +=",
     "for (int c = 0; c < H - 1; ++c)\n                acc +="),
    ("awq natural nibble order", "{0, 2, 4, 6, 1, 3, 5, 7};", "{0, 1, 2, 3, 4, 5, 6, 7};"),
    ("awq qweight indexed as [N/8][K]", "aq[((size_t)e * K + kk) * (N / 8) + n / 8];",
     "aq[((size_t)e * (N / 8) + n / 8) * K + kk];"),
    ("awq zero word of column ignored", "az[((size_t)e * (K / 32) + kk / 32) * (N / 8) + n / 8];",
     "az[((size_t)e * (K / 32) + kk / 32) * (N / 8)];"),
    ("awq scales not transposed", "as[((size_t)e * (K / 32) + kk / 32) * N + n];",
     "as[((size_t)e * N + n) * (K / 32) + kk / 32];"),
    ("imported zero nibble by column of K", "r % 8,\n                           oracle_awq_z",
     "kk % 8,\n                           oracle_awq_z"),
    ("imported rows not offset", "int r = row0 + n;", "int r = n;"),
]

RA_CHECKS = [
    ra.test_router_logits_exact_on_tiny_input,
    ra.test_router_logits_one_hot_picks_a_column,
    ra.test_router_logits_match_library_product,
    ra.test_awq_order_word_gives_column_index,
    ra.test_awq_single_nibbles_land_where_derived,
    ra.test_awq_scales_are_transposed,
    ra.test_awq_import_preserves_every_dequantised_weight,
    ra.test_awq_import_into_upper_half_leaves_lower_half,
]


@pytest.mark.parametrize("name,orig,mut", RA_MUTANTS, ids=[m[0] for m in RA_MUTANTS])
def test_planted_router_awq_mistake_is_caught(tmp_path, name, orig, mut):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for '{name}' not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(orig, mut))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fvisibility=hidden", str(mpath), "-o", str(lib), "-lm"])
    caught = []
    with oracle.using_library(str(lib)):
        for check in RA_CHECKS:
            try:
                check(oracle)
            except (AssertionError, IndexError, ValueError):
                caught.append(check)
    assert caught, f"no pin rejects the planted mistake '{name}'"


def test_unmutated_source_passes_every_check():
    for check in CHECKS + NVFP4_CHECKS + RA_CHECKS:
        check(oracle)
    assert inputs.TINY.shape.k == 2
