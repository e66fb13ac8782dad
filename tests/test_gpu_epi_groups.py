"""The two-group epilogue (two groups of four warps taking alternate tiles
whole, four TMEM buffers) against the one-group epilogue, on the layers it
is chosen for: 64-wide tiles, short and long reductions.
Every output must be bit-identical either way (each row gets the same
accumulators and the same epilogue arithmetic) and, on integer data, equal
to the oracle.  The cases include strided dgrad with residue classes that
have no taps (units without accumulators, which the groups also share),
odd tile counts, int8 dgrad and the Winograd transform-domain GEMM."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import assert_exact, device_ok, f64, guarded_empty, inputs, problem, to_f64

pytestmark = pytest.mark.gpu


def _both(fn):
    out = {}
    try:
        for mode in (1, 2):
            igc.igconv_set_tuning(igc.TUNE_EPI_GROUPS, mode)
            out[mode] = fn()
    finally:
        igc.igconv_set_tuning(igc.TUNE_EPI_GROUPS, 0)
    np.testing.assert_array_equal(out[1], out[2])
    return out[2]


def _dgrad(pb, inp, fmt):
    dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]),
                              torch.float16 if fmt == "f16" else torch.bfloat16, "cuda")
    igc.conv2d_dgrad(pb, dX.dtype, inp["dY"].cuda(), inp["W"].cuda(), None, dX)
    device_ok()
    check()
    return to_f64(dX)


def _fprop(pb, inp, fmt):
    P, Q = igc.conv2d_output_size(pb)
    Y, check = guarded_empty((pb["N"], P, Q, pb["K"]),
                             torch.float16 if fmt == "f16" else torch.bfloat16, "cuda")
    igc.conv2d_fprop(pb, Y.dtype, inp["X"].cuda(), inp["W"].cuda(), inp["bias"].cuda(), None, Y,
                     1.0, 0.0, True)
    device_ok()
    check()
    return to_f64(Y)


DGRAD = [
    problem(4, 23, 21, 64, 64, 3, 3, (1, 1), (2, 2)),      # 4 residue classes, 1-4 taps
    problem(2, 17, 19, 64, 48, 3, 3, (0, 0), (4, 4)),      # stride 4: classes with no taps
    problem(3, 15, 13, 64, 256, 1, 1),                     # 1x1: four blocks per tile
    problem(1, 9, 11, 48, 64, 1, 1, (0, 0), (2, 2)),       # 1x1 strided: uncovered rows
    problem(2, 20, 18, 64, 128, 3, 3, (1, 1)),             # stride 1, 18 blocks per tile
]


@pytest.mark.parametrize("pb", DGRAD, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS")
                         + f"_s{p['stride_h']}")
def test_epi_groups_dgrad_bit_identical_and_exact(pb):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 91)
    got = _both(lambda: _dgrad(pb, inp, "f16"))
    assert_exact(got, oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"])), "f16", "dgrad")
    rinp, _, _ = inputs(pb, "bf16", "normal_he", 92)
    _both(lambda: _dgrad(pb, rinp, "bf16"))


@pytest.mark.parametrize("pb", [problem(3, 14, 15, 64, 64, 1, 1),
                                problem(2, 13, 11, 128, 64, 1, 1)],
                         ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_epi_groups_fprop_bit_identical_and_exact(pb):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 93, bias=True)
    got = _both(lambda: _fprop(pb, inp, "f16"))
    ref = oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True)
    assert_exact(got, ref, "f16", "fprop")


def test_epi_groups_int8_dgrad_bit_identical_and_exact():
    pb = problem(2, 11, 9, 64, 48, 3, 3, (1, 1), (2, 1))
    inp, P, Q = inputs(pb, "i8", "int8", 94)
    need = igc.conv2d_dgrad_int8_workspace_size(pb)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def run():
        dX = torch.empty((pb["N"], pb["H"], pb["W"], pb["C"]), dtype=torch.int32, device="cuda")
        igc.conv2d_dgrad_int8(pb, inp["dY"].cuda(), inp["W"].cuda(), dX, ws)
        device_ok()
        return dX.cpu().numpy()
    got = _both(run)
    np.testing.assert_array_equal(got, oracle.dgrad_int8(pb, inp["dY"].numpy(), inp["W"].numpy()))


def test_epi_groups_winograd_bit_identical():
    pb = problem(2, 13, 11, 48, 64, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "bf16", "normal_he", 95, bias=True)
    need = igc.conv2d_fprop_winograd_workspace_size(pb, torch.bfloat16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def run():
        Y = torch.empty((pb["N"], P, Q, pb["K"]), dtype=torch.bfloat16, device="cuda")
        igc.conv2d_fprop_winograd(pb, torch.bfloat16, inp["X"].cuda(), inp["W"].cuda(),
                                  inp["bias"].cuda(), None, Y, relu=True, workspace=ws)
        device_ok()
        return to_f64(Y)
    _both(run)
