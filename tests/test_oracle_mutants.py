"""Planted mistakes: each mutant is a copy of the oracle's C source with one
plausible slip, compiled on the CPU.  The pins must reject every mutant,
which shows they constrain the parts of the oracle the GPU parity tests rely
on.  The real oracle is never modified."""
import os
import subprocess

import numpy as np
import pytest

import oracle as oracle_mod
from tests import test_oracle_3d_pins as pins3d
from tests import test_oracle_abs_pins as apins
from tests import test_oracle_grouped_pins as gpins
from tests import test_oracle_int8_back_pins as i8pins
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle_mod.__file__), "conv_oracle.c")

# (name, text to find, replacement, occurrence index among matches)
MUTANTS = [
    ("fprop pad sign", "int h = pp * p->stride_h - p->pad_h + r * p->dil_h;",
     "int h = pp * p->stride_h + p->pad_h + r * p->dil_h;", 0),
    ("fprop dilation dropped", "int w = q * p->stride_w - p->pad_w + s * p->dil_w;",
     "int w = q * p->stride_w - p->pad_w + s;", 0),
    ("fprop filter taps transposed",
     "double f = t->Wt[(((int64_t)k * p->R + r) * p->S + s) * p->C + c];",
     "double f = t->Wt[(((int64_t)k * p->R + s % p->R) * p->S + r % p->S) * p->C + c];", 0),
    ("fprop bias dropped", "if (t->bias) v += t->bias[k];", "", 0),
    ("fprop relu before bias", "    if (t->bias) v += t->bias[k];\n    if (t->relu && v < 0.0) v = 0.0;",
     "    if (t->relu && v < 0.0) v = 0.0;\n    if (t->bias) v += t->bias[k];", 0),
    ("fprop beta scaled by alpha", "if (t->beta != 0.0) v += t->beta * t->Cin[e];",
     "if (t->beta != 0.0) v += t->alpha * t->beta * t->Cin[e];", 0),
    ("dgrad stride test dropped", "if (th < 0 || th % p->stride_h != 0) continue;",
     "if (th < 0) continue;", 0),
    ("dgrad flipped tap", "int th = h + p->pad_h - r * p->dil_h;",
     "int th = h + p->pad_h - (p->R - 1 - r) * p->dil_h;", 0),
    ("dgrad uses wrong weight channel",
     "double f = t->Wt[(((int64_t)k * p->R + r) * p->S + s) * p->C + c];",
     "double f = t->Wt[(((int64_t)(k % p->C) * p->R + r) * p->S + s) * p->C + (c % p->K)];", 1),
    ("wgrad dilation sign", "int w = q * p->stride_w - p->pad_w + s * p->dil_w;",
     "int w = q * p->stride_w - p->pad_w - s * p->dil_w + 2 * s;", 1),
    ("wgrad drops last image", "for (int n = 0; n < p->N; ++n) {\n        for (int pp = 0; pp < t->P; ++pp) {",
     "for (int n = 0; n < p->N - 1; ++n) {\n        for (int pp = 0; pp < t->P; ++pp) {", 0),
    ("out size off by one", "return (int)(span / stride) + 1;", "return (int)((span + 1) / stride) + 1;", 0),
    ("rounding half up", "double units = nearbyint(a / quantum);", "double units = floor(a / quantum + 0.5);", 0),
    ("requant half away from zero", "double y = nearbyint(prod);", "double y = round(prod);", 0),
    ("requant no saturation", "if (y > 127.0) y = 127.0;", "", 0),
    ("requant multiplier from fp32 scales", "double m = act_scale * w_scale / out_scale;",
     "double m = (double)(float)act_scale * (double)(float)w_scale / (double)(float)out_scale;", 0),
    ("int8 bias dropped", "int64_t v = sum + (t->bias ? (int64_t)t->bias[k] : 0);", "int64_t v = sum;", 0),
    ("grouped fprop group from k mod G", "int g = k / t->Kg;", "int g = k % t->G;", 0),
    ("grouped fprop channel order reversed in group",
     "double f = t->B_in[(((int64_t)k * p->R + r) * p->S + s) * t->Cg + jj];",
     "double f = t->B_in[(((int64_t)k * p->R + r) * p->S + s) * t->Cg + (t->Cg - 1 - jj)];", 0),
    ("grouped dgrad sums every output channel",
     "for (int k = g * t->Kg; k < (g + 1) * t->Kg; ++k) {", "for (int k = 0; k < p->K; ++k) {", 0),
    ("grouped dgrad flipped tap", "int th = h + p->pad_h - r * p->dil_h;",
     "int th = h + p->pad_h - (p->R - 1 - r) * p->dil_h;", 1),
    ("grouped wgrad drops the group offset", "int c = (k / t->Kg) * t->Cg + jj;", "int c = jj;", 0),
    ("3d depth pad sign", "int d = o * p->stride_d - p->pad_d + tt * p->dil_d;",
     "int d = o * p->stride_d + p->pad_d + tt * p->dil_d;", 0),
    ("3d depth dilation dropped", "int d = o * p->stride_d - p->pad_d + tt * p->dil_d;",
     "int d = o * p->stride_d - p->pad_d + tt;", 0),
    ("3d filter depth index from r",
     "double f = t->Wt[((((int64_t)k * p->T + tt) * p->R + r) * p->S + s) * p->C + c];",
     "double f = t->Wt[((((int64_t)k * p->T + r % p->T) * p->R + tt % p->R) * p->S + s) * p->C + c];", 0),
    ("3d dgrad depth stride test dropped", "if (td < 0 || td % p->stride_d != 0) continue;",
     "if (td < 0) continue;", 0),
    ("3d wgrad depth dilation dropped", "int d = o * p->stride_d - p->pad_d + tt * p->dil_d;",
     "int d = o * p->stride_d - p->pad_d + tt;", 1),
    ("int8 dgrad flipped tap", "int th = h + p->pad_h - r * p->dil_h;",
     "int th = h + p->pad_h - (p->R - 1 - r) * p->dil_h;", 3),
    ("int8 dgrad stride test dropped", "if (th < 0 || th % p->stride_h != 0) continue;",
     "if (th < 0) continue;", 3),
    ("int8 wgrad dilation dropped", "int w = q * p->stride_w - p->pad_w + s * p->dil_w;",
     "int w = q * p->stride_w - p->pad_w + s;", 7),
    ("int8 backward saturates instead of wrapping",
     "uint32_t u = (uint32_t)((uint64_t)v & 0xFFFFFFFFu);",
     "if (v > 2147483647LL) v = 2147483647LL; if (v < -2147483647LL - 1) v = -2147483647LL - 1;"
     " uint32_t u = (uint32_t)((uint64_t)v & 0xFFFFFFFFu);", 0),
    ("int8 wgrad reads X at the dY channel",
     "int64_t x = t->A_in[(((int64_t)n * p->H + h) * p->W + w) * p->C + c];",
     "int64_t x = t->A_in[(((int64_t)n * p->H + h) * p->W + w) * p->C + k % p->C];", 0),
    ("permute swaps h and w", "int64_t di = (((int64_t)n * H + h) * W + w) * C + c;\n                    memcpy",
     "int64_t di = (((int64_t)n * W + w) * H + h) * C + c;\n                    memcpy", 0),
]

# Slips in the second output, A = |alpha| * sum |x*w| (the tolerance scale).
# Each entry is (name, [(text to find, replacement, occurrence), ...]); the
# edits are applied in order.  Occurrence i of the A store is pass i in source
# order: fprop, dgrad, wgrad, grouped fprop / dgrad / wgrad, 3D fprop / dgrad /
# wgrad.
A_STORE = "if (t->A) t->A[j] = fabs(t->alpha) * asum;"
_PASSES = ["fprop", "dgrad", "wgrad", "grouped fprop", "grouped dgrad", "grouped wgrad",
           "3d fprop", "3d dgrad", "3d wgrad"]
ABS_MUTANTS = [
    (f"{name} A of the signed sum", [(A_STORE, "if (t->A) t->A[j] = fabs(t->alpha * sum);", i)])
    for i, name in enumerate(_PASSES)
] + [
    (f"{name} A without |alpha|", [(A_STORE, "if (t->A) t->A[j] = asum;", i)])
    for i, name in enumerate(_PASSES)
] + [
    ("fprop A as a sum of magnitudes", [("asum += fabs(x * f);", "asum += fabs(x) + fabs(f);", 0)]),
    ("fprop A as a product of sums", [
        ("double sum = 0.0, asum = 0.0;", "double sum = 0.0, asum = 0.0, sx = 0.0, sf = 0.0;", 0),
        ("asum += fabs(x * f);", "sx += fabs(x); sf += fabs(f);", 0),
        (A_STORE, "asum = sx * sf; " + A_STORE, 0)]),
    ("dgrad A from the wrong input channel", [
        ("asum += fabs(g * f);",
         "asum += fabs(g * t->Wt[(((int64_t)k * p->R + r) * p->S + s) * p->C + (c + 1) % p->C]);",
         0)]),
    ("wgrad A from the previous image", [
        ("asum += fabs(g * x);",
         "asum += fabs(g * t->X[(((int64_t)((n + 1) % p->N) * p->H + h) * p->W + w) * p->C + c]);",
         0)]),
    ("grouped dgrad A over every output channel", [
        ("asum += fabs(gy * f);",
         "for (int k2 = 0; k2 < p->K; ++k2) asum += fabs(t->A_in[(((int64_t)n * t->P + pp) * t->Q"
         " + q) * p->K + k2] * f) / t->Kg;", 0)]),
    ("A includes the bias", [(A_STORE, "if (t->A) t->A[j] = fabs(t->alpha) * asum + "
                              "(t->bias ? fabs(t->bias[k]) : 0.0);", 0)]),
]

PIN_CALLS = [
    (pins.test_output_size_golden, {}),
    (pins.test_output_size_counts_valid_windows, {}),
    (pins.test_fprop_hand_examples, {}),
    (pins.test_fprop_epilogue_alpha_beta_bias_relu, {}),
    (pins.test_fprop_dilation_is_zero_inserted_filter, {}),
    (pins.test_backward_hand_example, {}),
    (pins.test_dgrad_uncovered_rows_are_zero, {}),
    (pins.test_dgrad_wgrad_alpha_beta, {}),
    (pins.test_requant_multiplier_is_fp32_of_double_quotient, {}),
    (pins.test_requant_exact_against_fractions, {}),
    (pins.test_requant_relu, {}),
    (pins.test_int8_matches_int64_einsum, {}),
    (pins.test_f16_bf16_hand_ties, {}),
    (pins.test_f16_rounding_matches_numpy, {}),
] + [(pins.test_fprop_brute_force_im2col, {"pb": pb}) for pb in [
    pins._pb(2, 7, 9, 3, 5, 3, 3, 1, 1, 1, 1, 1, 1),
    pins._pb(3, 10, 11, 2, 4, 5, 3, 2, 1, 3, 2, 2, 1),
]] + [(pins.test_adjoint_identities_exact, {"pb": pb}) for pb in pins.ADJOINT_PROBLEMS] \
  + [(pins.test_permutes_index_formula_and_round_trip, {"dtype": np.float16})] \
  + [(gpins.test_grouped_hand_example_with_multiplier, {})] \
  + [(pins3d.test_depth_one_is_2d, {})] \
  + [(pins3d.test_separable_filter_is_sum_of_2d, {"pb": pb}) for pb in pins3d.PROBLEMS_3D] \
  + [(pins3d.test_3d_adjoint_identities_exact, {"pb": pb}) for pb in pins3d.PROBLEMS_3D] \
  + [(gpins.test_grouped_is_dense_with_block_diagonal_filter, {"pb": pb, "groups": g})
     for pb, g in gpins.GROUPED_PROBLEMS] \
  + [(fn, {"pb": pb}) for pb in apins.PROBLEMS_2D
     for fn in (apins.test_fprop_abs_sum_is_im2col_of_magnitudes,
                apins.test_dgrad_abs_sum_is_col2im_of_magnitudes,
                apins.test_wgrad_abs_sum_is_im2col_of_magnitudes)] \
  + [(apins.test_grouped_abs_sums_are_torch_convs_of_magnitudes, {"pb": pb, "groups": g})
     for pb, g in gpins.GROUPED_PROBLEMS] \
  + [(apins.test_3d_abs_sums_are_torch_convs_of_magnitudes, {"pb": pb})
     for pb in pins3d.PROBLEMS_3D] \
  + [(fn, {"pb": pb}) for pb in i8pins.PROBLEMS
     for fn in (i8pins.test_int8_backward_equals_fp64_passes,
                i8pins.test_int8_backward_adjoint_identities_exact)] \
  + [(i8pins.test_int8_wgrad_wraps_past_2_31, {}), (i8pins.test_int8_dgrad_wraps_past_2_31, {})]


def _first_failing_pin():
    for fn, kw in PIN_CALLS:
        try:
            fn(oracle_mod, **kw)
        except (AssertionError, ValueError, IndexError):
            return fn.__name__
    return None


def test_mutant_catalogue_applies_to_current_source():
    src = open(SRC).read()
    for name, find, _, occ in MUTANTS:
        assert src.count(find) > occ, f"mutant '{name}' no longer matches the source"
    for name, edits in ABS_MUTANTS:
        for find, _, occ in edits:
            assert src.count(find) > occ, f"mutant '{name}' no longer matches the source"


def _apply(src, find, repl, occ):
    pos = -1
    for _ in range(occ + 1):
        pos = src.index(find, pos + 1)
    return src[:pos] + repl + src[pos + len(find):]


def _assert_rejected(tmp_path, name, mutated):
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-std=c11", "-D_GNU_SOURCE", "-shared",
                    "-fPIC", "-pthread", "-o", str(so_path), str(c_path), "-lm"], check=True)
    with oracle_mod.use_library(str(so_path)):
        caught = _first_failing_pin()
    assert caught is not None, f"no pin rejects the mutant '{name}'"


@pytest.mark.parametrize("name,find,repl,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, find, repl, occ):
    _assert_rejected(tmp_path, name, _apply(open(SRC).read(), find, repl, occ))


@pytest.mark.parametrize("name,edits", ABS_MUTANTS, ids=[m[0] for m in ABS_MUTANTS])
def test_pins_reject_abs_sum_mutant(tmp_path, name, edits):
    src = open(SRC).read()
    for find, repl, occ in edits:
        src = _apply(src, find, repl, occ)
    _assert_rejected(tmp_path, name, src)
