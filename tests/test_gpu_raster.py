"""Scheduling, staging and kernel-choice knobs that must not change a bit:
the tile raster order of the persistent scheduler (IGCONV_TUNE_RASTER, the
CUTLASS example's "Swizzling Stride"), the shared-memory-resident filter
(IGCONV_TUNE_RESIDENT_FILTER) and the kernels whose epilogue holds only the
16-bit store path (IGCONV_TUNE_EPILOGUE_KERNEL).  Every setting computes
every tile exactly once with the same reduction and epilogue arithmetic, so
outputs are bit-identical to the built-in setting (and exact against the
oracle on integer data)."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import assert_exact, device_ok, f64, inputs, problem, to_f64

pytestmark = pytest.mark.gpu

CASES = [
    # 64-wide tiles, ragged last row tile
    ("fprop", problem(2, 23, 21, 64, 64, 3, 3, (1, 1))),
    # 128-wide tiles on CTA pairs, three column tiles
    ("fprop", problem(2, 20, 19, 64, 384, 3, 3, (1, 1))),
    # strided dgrad: four residue-class sub-problems in one launch
    ("dgrad", problem(2, 19, 22, 64, 128, 3, 3, (1, 1), (2, 2))),
    # stride-1 dgrad, 128-wide tiles
    ("dgrad", problem(1, 30, 31, 128, 64, 3, 3, (1, 1))),
]


def run(kind, pb, inp):
    if kind == "fprop":
        return to_f64(igc.fprop(pb, inp["X"].cuda(), inp["W"].cuda(), bias=inp["bias"].cuda(),
                                relu=True))
    return to_f64(igc.dgrad(pb, inp["dY"].cuda(), inp["W"].cuda()))


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0] + "_" + "x".join(
    str(c[1][k]) for k in "NHWCK") + f"_s{c[1]['stride_h']}")
def test_raster_orders_bit_identical(case):
    kind, pb = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 61, bias=True)
    if kind == "fprop":
        ref = oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True)
    else:
        ref = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]))
    outs = {}
    try:
        for g in (0, 2, 3, 8, 64):
            igc.igconv_set_tuning(igc.TUNE_RASTER, g)
            outs[g] = run(kind, pb, inp)
            device_ok()
            assert_exact(outs[g], ref, "f16", f"{kind} raster {g}")
    finally:
        igc.igconv_set_tuning(igc.TUNE_RASTER, 0)
    for g, o in outs.items():
        assert np.array_equal(o, outs[0]), f"raster {g} differs from the built-in order"


# Resident filter (IGCONV_TUNE_RESIDENT_FILTER): 64-wide single-column plans
# with at most 4 reduction blocks keep the filter in shared memory; the
# MMAs read the same operands, so results are bit-identical either way.
RES_CASES = [
    ("fprop", problem(2, 21, 23, 64, 64, 2, 2, (1, 1))),        # 4 blocks: resident
    ("dgrad", problem(2, 19, 20, 64, 64, 2, 2, (1, 1))),        # stride-1 dgrad, 4 blocks
    ("fprop", problem(2, 21, 23, 64, 64, 3, 3, (1, 1))),        # 9 blocks: not resident
    ("dgrad", problem(2, 16, 17, 64, 256, 1, 1)),               # 1x1 dgrad: 4 blocks of K
    ("fprop", problem(2, 40, 42, 3, 64, 7, 7, (3, 3), (2, 2))),  # packed stem: 4 blocks
    ("fprop", problem(1, 15, 14, 128, 48, 3, 3, (1, 1))),       # 18 blocks: not resident
]


@pytest.mark.parametrize("case", RES_CASES, ids=lambda c: c[0] + "_" + "x".join(
    str(c[1][k]) for k in "NHWCKRS"))
def test_resident_filter_bit_identical(case):
    kind, pb = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 67, bias=True)
    if kind == "fprop":
        ref = oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True)
    else:
        ref = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]))
    outs = []
    try:
        for off in (0, 1):
            igc.igconv_set_tuning(igc.TUNE_RESIDENT_FILTER, off)
            outs.append(run(kind, pb, inp))
            device_ok()
            assert_exact(outs[-1], ref, "f16", f"{kind} resident filter off={off}")
    finally:
        igc.igconv_set_tuning(igc.TUNE_RESIDENT_FILTER, 0)
    assert np.array_equal(outs[0], outs[1])


# 16-bit-store epilogue kernels (IGCONV_TUNE_EPILOGUE_KERNEL = 0, the
# built-in choice) against the kernels that carry every epilogue (1), over
# each store form: 32- and 64-column boxes, CTA pairs, the resident filter,
# residue-class rows through the 5D view, per-row stores, beta * Cin.
EPI_CASES = [
    ("fprop", problem(2, 23, 21, 64, 64, 3, 3, (1, 1)), 0.0),       # 64-wide, two groups
    ("fprop", problem(2, 20, 19, 64, 384, 3, 3, (1, 1)), 0.0),      # 128-wide CTA pairs
    ("fprop", problem(2, 14, 15, 64, 256, 1, 1), 0.0),              # 256-wide, 64-column boxes
    ("fprop", problem(2, 21, 23, 64, 64, 2, 2, (1, 1)), -1.0),      # resident filter, beta
    ("dgrad", problem(2, 28, 56, 64, 64, 3, 3, (1, 1), (2, 2)), 0.0),   # 5D class rows
    ("dgrad", problem(2, 13, 12, 16, 24, 3, 3, (1, 1), (2, 2)), 2.0),   # per-row stores, beta
    ("fprop", problem(2, 40, 42, 3, 64, 7, 7, (3, 3), (2, 2)), 0.0),    # packed stem
]


def run_ab(kind, pb, inp, beta):
    if kind == "fprop":
        cin = inp["C_fprop"].cuda() if beta else None
        return to_f64(igc.fprop(pb, inp["X"].cuda(), inp["W"].cuda(), bias=inp["bias"].cuda(),
                                Cin=cin, beta=beta, relu=True))
    cin = inp["C_dgrad"].cuda() if beta else None
    return to_f64(igc.dgrad(pb, inp["dY"].cuda(), inp["W"].cuda(), Cin=cin, beta=beta))


@pytest.mark.parametrize("case", EPI_CASES, ids=lambda c: c[0] + "_" + "x".join(
    str(c[1][k]) for k in "NHWCKRS") + f"_s{c[1]['stride_h']}_b{c[2]:g}")
def test_store16_epilogue_kernels_bit_identical(case):
    kind, pb, beta = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 83, bias=True, cin=True)
    if kind == "fprop":
        ref = oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True,
                           Cin=f64(inp["C_fprop"]) if beta else None, beta=beta)
    else:
        ref = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]),
                           Cin=f64(inp["C_dgrad"]) if beta else None, beta=beta)
    outs = []
    try:
        for general in (0, 1):
            igc.igconv_set_tuning(igc.TUNE_EPILOGUE_KERNEL, general)
            outs.append(run_ab(kind, pb, inp, beta))
            device_ok()
            assert_exact(outs[-1], ref, "f16", f"{kind} general epilogue={general}")
    finally:
        igc.igconv_set_tuning(igc.TUNE_EPILOGUE_KERNEL, 0)
    assert np.array_equal(outs[0], outs[1])
