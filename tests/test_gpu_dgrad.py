"""GPU parity of conv2d_dgrad against the oracle, including the stride
decomposition (one sub-convolution per output residue class, with classes
that have no taps and input rows no output reads)."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import WORKLOADS
from tests.helpers import (assert_close, assert_exact, device_ok, f64, guarded_empty, inputs,
                           problem, to_f64)

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16}


def run_dgrad(pb, inp, dtype, alpha=1.0, beta=0.0):
    dY, Wt = inp["dY"].cuda(), inp["W"].cuda()
    Cin = inp["C_dgrad"].cuda() if beta != 0.0 else None
    dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]), FMT[dtype], "cuda")
    igc.conv2d_dgrad(pb, FMT[dtype], dY, Wt, Cin, dX, alpha, beta)
    device_ok()
    check()
    return to_f64(dX)


def oracle_dgrad(pb, inp, alpha=1.0, beta=0.0):
    return oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]),
                        Cin=f64(inp["C_dgrad"]) if beta != 0.0 else None, alpha=alpha, beta=beta,
                        want_abs=True)


@pytest.mark.parametrize("name", ["tiny", "cutlass_notebook"])
def test_page_workloads_bit_exact(name):
    wl = WORKLOADS[name]
    pb = wl["problem"]
    inp, P, Q = inputs(pb, wl["dtype"], wl["recipe"], wl["seed"], cin=True)
    for alpha, beta in [(1.0, 0.0), (1.0, 1.0), (-2.0, 0.5)]:
        got = run_dgrad(pb, inp, "f16", alpha, beta)
        ref, _ = oracle_dgrad(pb, inp, alpha, beta)
        assert_exact(got, ref, "f16", f"{name} alpha={alpha} beta={beta}")


SHAPES = [
    problem(1, 4, 4, 64, 64, 1, 1),
    problem(2, 9, 11, 24, 40, 3, 3, (1, 1)),
    problem(2, 12, 12, 32, 16, 3, 3, (2, 2), (1, 1), (2, 2)),     # dilation
    problem(2, 13, 12, 16, 24, 3, 3, (1, 1), (2, 2)),             # stride 2, odd H
    problem(1, 17, 16, 8, 8, 2, 2, (0, 0), (3, 3)),               # stride > R: rows nobody reads
    problem(2, 10, 9, 16, 32, 3, 5, (1, 2), (2, 3), (2, 1)),      # stride + dilation mix
    problem(1, 15, 15, 8, 8, 7, 7, (3, 3), (2, 2)),
    problem(2, 8, 8, 72, 136, 3, 3, (1, 1)),                      # ragged channel blocks
    problem(2, 14, 14, 16, 16, 1, 1, (0, 0), (2, 2)),             # strided 1x1
    problem(2, 9, 9, 16, 16, 3, 3, (1, 1), (4, 4)),               # 16 residue classes
]


@pytest.mark.parametrize("pb", SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS") +
                         f"_p{p['pad_h']}{p['pad_w']}_s{p['stride_h']}{p['stride_w']}"
                         f"_d{p['dil_h']}{p['dil_w']}")
def test_shapes_integer_exact(pb):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 13, cin=True)
    got = run_dgrad(pb, inp, "f16")
    ref, _ = oracle_dgrad(pb, inp)
    assert_exact(got, ref, "f16", "integer dgrad")
    got = run_dgrad(pb, inp, "f16", 1.0, 2.0)
    ref, _ = oracle_dgrad(pb, inp, 1.0, 2.0)
    assert_exact(got, ref, "f16", "integer dgrad with beta")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("pb", [SHAPES[1], SHAPES[3], SHAPES[5]],
                         ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_shapes_random_normal(pb, dtype):
    inp, P, Q = inputs(pb, dtype, "normal_he", 17)
    got = run_dgrad(pb, inp, dtype)
    ref, A = oracle_dgrad(pb, inp)
    assert_close(got, ref, A, dtype, "normal dgrad")


def test_knobs_keep_results():
    """Tile widths 64 and 128 add a tile's blocks in the same two
    accumulators when 64-wide tiles are not given one issuer per tile
    (IGCONV_TUNE_ONE_ISSUER = 1), so they agree bit for bit; with one
    accumulator per tile (the built-in choice for these short residue-class
    reductions) the sums round differently but stay within the bound."""
    pb = problem(2, 14, 14, 256, 64, 3, 3, (1, 1), (2, 2))
    inp, P, Q = inputs(pb, "bf16", "normal_he", 19)
    ref, A = oracle_dgrad(pb, inp)
    base = run_dgrad(pb, inp, "bf16")                  # the planner's own width
    assert_close(base, ref, A, "bf16", "default")
    got = {}
    try:
        for key, val in [(igc.TUNE_BLOCK_N, 64), (igc.TUNE_BLOCK_N, 128), (igc.TUNE_MAX_CTAS, 3)]:
            igc.igconv_set_tuning(key, val)
            got[(key, val)] = run_dgrad(pb, inp, "bf16")
            assert_close(got[(key, val)], ref, A, "bf16", f"knob {key}={val}")
            if (key, val) == (igc.TUNE_BLOCK_N, 64):
                igc.igconv_set_tuning(igc.TUNE_ONE_ISSUER, 1)
                got["two_acc"] = run_dgrad(pb, inp, "bf16")
                igc.igconv_set_tuning(igc.TUNE_ONE_ISSUER, 0)
            igc.igconv_set_tuning(key, 0)
    finally:
        igc.igconv_set_tuning(igc.TUNE_BLOCK_N, 0)
        igc.igconv_set_tuning(igc.TUNE_MAX_CTAS, 0)
        igc.igconv_set_tuning(igc.TUNE_ONE_ISSUER, 0)
    np.testing.assert_array_equal(got["two_acc"], got[(igc.TUNE_BLOCK_N, 128)])
    np.testing.assert_array_equal(got[(igc.TUNE_MAX_CTAS, 3)], base)


# Stride-1 dgrad with 128 input channels runs on CTA pairs; odd row-tile
# counts leave the last pair's second CTA without rows.
PAIR_SHAPES = [
    problem(2, 15, 15, 128, 64, 3, 3, (1, 1)),      # 4 row tiles
    problem(1, 23, 23, 128, 32, 3, 3, (1, 1)),      # 5 row tiles
    problem(2, 14, 14, 256, 96, 3, 3, (2, 2), (1, 1), (2, 2)),   # dilation 2
]


@pytest.mark.parametrize("pb", PAIR_SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_cta_pairs_bit_identical(pb):
    inp, P, Q = inputs(pb, "bf16", "normal_he", 31)
    iinp, _, _ = inputs(pb, "f16", "int_uniform", 37)
    iref, _ = oracle_dgrad(pb, iinp)
    ref, A = oracle_dgrad(pb, inp)
    paired = run_dgrad(pb, inp, "bf16")
    assert_close(paired, ref, A, "bf16", "pairs")
    assert_exact(run_dgrad(pb, iinp, "f16"), iref, "f16", "integer, pairs")
    try:
        igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 1)
        single = run_dgrad(pb, inp, "bf16")
        assert_exact(run_dgrad(pb, iinp, "f16"), iref, "f16", "integer, no pairs")
    finally:
        igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 0)
    np.testing.assert_array_equal(paired, single)


PAIR256_SHAPES = [
    problem(2, 14, 14, 256, 128, 3, 3, (1, 1)),     # 4 row tiles
    problem(1, 23, 23, 320, 64, 3, 3, (1, 1)),      # 5 row tiles, C ragged in tile 2
]


@pytest.mark.parametrize("pb", PAIR256_SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_cta_pairs_256_bit_identical(pb):
    """256-wide tiles on CTA pairs (tuning value 2) against single CTAs."""
    inp, P, Q = inputs(pb, "bf16", "normal_he", 53)
    iinp, _, _ = inputs(pb, "f16", "int_uniform", 59)
    iref, _ = oracle_dgrad(pb, iinp)
    ref, A = oracle_dgrad(pb, inp)
    out = {}
    try:
        igc.igconv_set_tuning(igc.TUNE_BLOCK_N, 256)
        for mode in (2, 1):
            igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, mode)
            out[mode] = run_dgrad(pb, inp, "bf16")
            assert_close(out[mode], ref, A, "bf16", f"pairs mode {mode}")
            assert_exact(run_dgrad(pb, iinp, "f16"), iref, "f16", f"integer, pairs mode {mode}")
    finally:
        igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 0)
        igc.igconv_set_tuning(igc.TUNE_BLOCK_N, 0)
    np.testing.assert_array_equal(out[2], out[1])
