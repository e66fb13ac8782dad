"""GPU parity of conv2d_fprop against the oracle.

Integer-valued fp16 inputs (the CUTLASS example's recipe) make every fp32
partial sum exact, so those outputs must equal the oracle rounded to fp16,
bit for bit.  Random-normal inputs are held to the acceptance tolerance and
to a per-element bound.  Tuning knobs must not change a single bit."""
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


def run_fprop(pb, inp, dtype, bias=False, beta=0.0, alpha=1.0, relu=False):
    P, Q = igc.conv2d_output_size(pb)
    X, Wt = inp["X"].cuda(), inp["W"].cuda()
    b = inp["bias"].cuda() if bias else None
    Cin = inp["C_fprop"].cuda() if beta != 0.0 else None
    Y, check = guarded_empty((pb["N"], P, Q, pb["K"]), FMT[dtype], "cuda")
    igc.conv2d_fprop(pb, FMT[dtype], X, Wt, b, Cin, Y, alpha, beta, relu)
    device_ok()
    check()
    return to_f64(Y)


def oracle_fprop(pb, inp, bias=False, beta=0.0, alpha=1.0, relu=False):
    return oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]) if bias else None,
                        Cin=f64(inp["C_fprop"]) if beta != 0.0 else None, alpha=alpha, beta=beta,
                        relu=relu, want_abs=True)


@pytest.mark.parametrize("name", ["tiny", "cutlass_notebook"])
def test_page_workloads_bit_exact(name):
    wl = WORKLOADS[name]
    pb = wl["problem"]
    inp, P, Q = inputs(pb, wl["dtype"], wl["recipe"], wl["seed"], bias=True, cin=True)
    for bias, relu, alpha, beta in [(False, False, 1.0, 0.0), (True, True, 1.0, 0.0),
                                    (True, False, 2.0, -1.0)]:
        got = run_fprop(pb, inp, "f16", bias=bias, relu=relu, alpha=alpha, beta=beta)
        ref, _ = oracle_fprop(pb, inp, bias=bias, relu=relu, alpha=alpha, beta=beta)
        assert_exact(got, ref, "f16", f"{name} bias={bias} relu={relu} beta={beta}")


# Shapes with ragged M tails, channel counts that are not multiples of 64,
# K not a multiple of the tile, strides, dilations, rectangular filters.
SHAPES = [
    problem(1, 4, 4, 64, 64, 1, 1),                               # a plain GEMM, one tile
    problem(2, 9, 7, 16, 24, 1, 1),                               # 1x1, ragged
    problem(3, 11, 13, 24, 40, 3, 5, (1, 2), (2, 1), (1, 2)),
    problem(2, 10, 10, 72, 136, 3, 3, (1, 1), (1, 1)),            # 2 channel blocks, K ragged
    problem(1, 15, 17, 8, 8, 7, 7, (3, 3), (2, 2)),               # stem-like
    problem(4, 6, 6, 128, 256, 3, 3, (1, 1)),                     # BN 256
    problem(2, 12, 12, 32, 64, 3, 3, (2, 2), (1, 1), (2, 2)),     # dilation 2
    problem(1, 3, 3, 16, 16, 3, 3),                               # P = Q = 1
    problem(2, 20, 3, 8, 16, 5, 1, (2, 0), (3, 1)),
    problem(1, 5, 5, 16, 1096, 1, 1),                             # bias too long to stage in smem
]


@pytest.mark.parametrize("pb", SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS") +
                         f"_p{p['pad_h']}{p['pad_w']}_s{p['stride_h']}{p['stride_w']}"
                         f"_d{p['dil_h']}{p['dil_w']}")
def test_shapes_integer_exact(pb):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 7, bias=True)
    got = run_fprop(pb, inp, "f16", bias=True)
    ref, _ = oracle_fprop(pb, inp, bias=True)
    assert_exact(got, ref, "f16", "integer fprop")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("pb", SHAPES[2:6], ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_shapes_random_normal(pb, dtype):
    inp, P, Q = inputs(pb, dtype, "normal_he", 11, bias=True, cin=True)
    got = run_fprop(pb, inp, dtype, bias=True, relu=True, beta=0.5, alpha=1.5)
    ref, A = oracle_fprop(pb, inp, bias=True, relu=True, beta=0.5, alpha=1.5)
    assert_close(got, ref, A, dtype, "normal fprop")


def test_knobs_keep_results():
    """Grid caps and tile widths 64/128 (same reduction grouping) leave every
    bit unchanged; width 256 groups the fp32 sums differently, so it agrees
    within tolerance, and exactly on integer data."""
    pb = problem(3, 14, 14, 64, 256, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "bf16", "normal_he", 3, bias=True)
    ref, A = oracle_fprop(pb, inp, bias=True)
    iinp, _, _ = inputs(pb, "f16", "int_uniform", 4, bias=True)
    iref, _ = oracle_fprop(pb, iinp, bias=True)
    results = {}
    try:
        for key, val in [(igc.TUNE_BLOCK_N, 64), (igc.TUNE_BLOCK_N, 128), (igc.TUNE_BLOCK_N, 256),
                         (igc.TUNE_MAX_CTAS, 1), (igc.TUNE_MAX_CTAS, 7)]:
            igc.igconv_set_tuning(key, val)
            got = run_fprop(pb, inp, "bf16", bias=True)
            assert_close(got, ref, A, "bf16", f"knob {key}={val}")
            assert_exact(run_fprop(pb, iinp, "f16", bias=True), iref, "f16", f"int knob {key}={val}")
            igc.igconv_set_tuning(key, 0)
            results[(key, val)] = got
    finally:
        igc.igconv_set_tuning(igc.TUNE_BLOCK_N, 0)
        igc.igconv_set_tuning(igc.TUNE_MAX_CTAS, 0)
    np.testing.assert_array_equal(results[(igc.TUNE_BLOCK_N, 64)], results[(igc.TUNE_BLOCK_N, 128)])
    base = run_fprop(pb, inp, "bf16", bias=True)      # the planner's own width
    assert (np.array_equal(base, results[(igc.TUNE_BLOCK_N, 128)])
            or np.array_equal(base, results[(igc.TUNE_BLOCK_N, 256)]))
    np.testing.assert_array_equal(results[(igc.TUNE_MAX_CTAS, 1)], base)
    np.testing.assert_array_equal(results[(igc.TUNE_MAX_CTAS, 7)], base)


def test_repeat_runs_identical():
    pb = problem(2, 28, 28, 64, 128, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "f16", "normal_he", 5)
    a = run_fprop(pb, inp, "f16")
    b = run_fprop(pb, inp, "f16")
    np.testing.assert_array_equal(a, b)


def test_cin_aliasing_output():
    # Cin == Y is allowed: each element is read before it is written
    pb = problem(2, 8, 8, 16, 32, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "f16", "int_uniform", 9, cin=True)
    Y = inp["C_fprop"].cuda().clone()
    igc.conv2d_fprop(pb, torch.float16, inp["X"].cuda(), inp["W"].cuda(), None, Y, Y, 1.0, 1.0,
                     False)
    device_ok()
    ref = oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), Cin=f64(inp["C_fprop"]), beta=1.0)
    assert_exact(to_f64(Y), ref, "f16", "Cin aliasing Y")


# Shapes whose fprop runs on CTA pairs (128-wide tiles, two or more row
# tiles), with odd row-tile counts so that the last pair's second CTA has no
# rows at all, and ragged K.
PAIR_SHAPES = [
    problem(2, 28, 28, 64, 128, 3, 3, (1, 1)),      # 13 row tiles
    problem(3, 11, 13, 24, 120, 3, 5, (1, 2), (2, 1), (1, 2)),
    problem(1, 19, 19, 72, 128, 3, 3, (1, 1)),      # 3 row tiles, 2 channel blocks
    problem(4, 16, 16, 64, 104, 1, 1),              # K ragged within the tile
]


@pytest.mark.parametrize("pb", PAIR_SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_cta_pairs_bit_identical(pb):
    """CTA pairs (256-row MMAs over two SMs) change no bit: each output row
    gets the same MMAs in the same order either way."""
    inp, P, Q = inputs(pb, "bf16", "normal_he", 23, bias=True)
    iinp, _, _ = inputs(pb, "f16", "int_uniform", 29, bias=True)
    iref, _ = oracle_fprop(pb, iinp, bias=True)
    ref, A = oracle_fprop(pb, inp, bias=True, relu=True)
    paired = run_fprop(pb, inp, "bf16", bias=True, relu=True)
    assert_close(paired, ref, A, "bf16", "pairs")
    assert_exact(run_fprop(pb, iinp, "f16", bias=True), iref, "f16", "integer, pairs")
    try:
        igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 1)
        single = run_fprop(pb, inp, "bf16", bias=True, relu=True)
        assert_exact(run_fprop(pb, iinp, "f16", bias=True), iref, "f16", "integer, no pairs")
    finally:
        igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 0)
    np.testing.assert_array_equal(paired, single)


# 256-wide tiles on CTA pairs (tuning value 2): odd row-tile counts and a
# ragged second column tile.
PAIR256_SHAPES = [
    problem(2, 14, 14, 128, 256, 3, 3, (1, 1)),     # 4 row tiles
    problem(1, 23, 23, 64, 320, 3, 3, (1, 1)),      # 5 row tiles, K ragged in tile 2
]


@pytest.mark.parametrize("pb", PAIR256_SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_cta_pairs_256_bit_identical(pb):
    inp, P, Q = inputs(pb, "bf16", "normal_he", 43, bias=True)
    iinp, _, _ = inputs(pb, "f16", "int_uniform", 47, bias=True)
    iref, _ = oracle_fprop(pb, iinp, bias=True)
    ref, A = oracle_fprop(pb, inp, bias=True, relu=True)
    out = {}
    try:
        igc.igconv_set_tuning(igc.TUNE_BLOCK_N, 256)
        for mode in (2, 1):
            igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, mode)
            out[mode] = run_fprop(pb, inp, "bf16", bias=True, relu=True)
            assert_close(out[mode], ref, A, "bf16", f"pairs mode {mode}")
            assert_exact(run_fprop(pb, iinp, "f16", bias=True), iref, "f16",
                         f"integer, pairs mode {mode}")
    finally:
        igc.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 0)
        igc.igconv_set_tuning(igc.TUNE_BLOCK_N, 0)
    np.testing.assert_array_equal(out[2], out[1])


# Few input channels (C <= 8): the first layer of a CNN.  Two paths: at
# dilation 1 (and stride_h * stride_w * C <= 64) the pixels are packed by
# space-to-depth into a padded image read as 128-byte windows of consecutive
# packed pixels; otherwise (or with IGCONV_TUNE_FEW_CHANNELS = 1) pixels are
# copied to 8-channel rows and a reduction block packs 8 taps x 8 channels.
FEW_SHAPES = [
    problem(2, 32, 32, 3, 64, 7, 7, (3, 3), (2, 2)),             # stem: 7x7 stride 2
    problem(1, 17, 13, 1, 16, 3, 3, (1, 1)),                      # one channel, ragged M
    problem(3, 15, 15, 4, 40, 5, 5, (4, 4), (1, 1), (2, 2)),      # dilation 2, 25 taps
    problem(2, 9, 11, 8, 136, 3, 3, (1, 1), (2, 1)),              # C = 8, K past one tile
    problem(1, 6, 6, 3, 8, 1, 1),                                 # 1x1, one padded block
    problem(2, 40, 44, 3, 64, 11, 11, (2, 2), (4, 4)),            # 11x11 stride 4: 64-ch pixels
    problem(2, 32, 32, 3, 96, 4, 4, (0, 0), (4, 4)),              # 4x4 patches, stride 4
    problem(1, 19, 23, 4, 32, 9, 9, (4, 4)),                      # 9 taps along w: 2 windows
    problem(2, 21, 20, 7, 24, 3, 5, (1, 2), (2, 3)),              # strides 2 x 3, 7 channels
    problem(1, 17, 16, 2, 8, 2, 2, (0, 0), (3, 3)),               # stride 3 > R
    problem(2, 13, 12, 5, 16, 3, 3, (3, 0), (1, 2)),              # pad 3 > R - 1
]
FEW_PATHS = {0: "packed", 1: "taps"}


@pytest.mark.parametrize("mode", FEW_PATHS, ids=FEW_PATHS.get)
@pytest.mark.parametrize("pb", FEW_SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS") +
                         f"_s{p['stride_h']}{p['stride_w']}_d{p['dil_h']}{p['dil_w']}")
def test_few_channels(pb, mode):
    try:
        igc.igconv_set_tuning(igc.TUNE_FEW_CHANNELS, mode)
        _few_channels_case(pb)
    finally:
        igc.igconv_set_tuning(igc.TUNE_FEW_CHANNELS, 0)


def _few_channels_case(pb):
    P, Q = igc.conv2d_output_size(pb)
    assert igc.conv2d_fprop_workspace_size(pb, torch.float16) > 0
    iinp, _, _ = inputs(pb, "f16", "int_uniform", 41, bias=True)
    iref, _ = oracle_fprop(pb, iinp, bias=True)
    got = to_f64(igc.fprop(pb, iinp["X"].cuda(), iinp["W"].cuda(), bias=iinp["bias"].cuda()))
    device_ok()
    assert_exact(got, iref, "f16", "integer few-channel fprop")
    inp, _, _ = inputs(pb, "bf16", "normal_he", 43, bias=True, cin=True)
    ref, A = oracle_fprop(pb, inp, bias=True, relu=True, alpha=1.5, beta=0.5)
    got = to_f64(igc.fprop(pb, inp["X"].cuda(), inp["W"].cuda(), bias=inp["bias"].cuda(),
                           Cin=inp["C_fprop"].cuda(), alpha=1.5, beta=0.5, relu=True))
    device_ok()
    assert_close(got, ref, A, "bf16", "normal few-channel fprop")


def test_few_channels_needs_workspace():
    pb = FEW_SHAPES[0]
    P, Q = igc.conv2d_output_size(pb)
    X = torch.zeros(pb["N"] * pb["H"] * pb["W"] * pb["C"], dtype=torch.float16, device="cuda")
    Wt = torch.zeros(pb["K"] * pb["R"] * pb["S"] * pb["C"], dtype=torch.float16, device="cuda")
    Y = torch.empty(pb["N"] * P * Q * pb["K"], dtype=torch.float16, device="cuda")
    with pytest.raises(igc.IgconvError, match="WORKSPACE"):
        igc.conv2d_fprop(pb, torch.float16, X, Wt, None, None, Y)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(igc.IgconvError, match="WORKSPACE"):
        igc.conv2d_fprop_ws(pb, torch.float16, X, Wt, None, None, Y, workspace=small)
