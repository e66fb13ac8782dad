"""GPU parity of strided dgrad on padded residue-class rows.

When H and W divide by the strides, every residue class of the stride
decomposition has the same H/stride_h x W/stride_w grid.  The library then
pads each class row to a multiple of 32 grid columns (when that adds at most
a sixth), so one epilogue warp's 32 rows are one class row of dX, written by
one TMA store through a 5D view of dX; the padding columns read zeros and
their results are clipped away.  IGCONV_TUNE_DGRAD_ROWS = 1 turns this off
(every output pixel stored by its own address).  Both settings must match
the oracle exactly on integer-valued data, and each other bit for bit on
random data.
"""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
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


def both_settings(fn):
    """fn() with padded rows (the built-in choice) and with row stores."""
    out = {}
    try:
        for mode in (0, 1):
            igc.igconv_set_tuning(igc.TUNE_DGRAD_ROWS, mode)
            out[mode] = fn()
    finally:
        igc.igconv_set_tuning(igc.TUNE_DGRAD_ROWS, 0)
    return out


def _id(p):
    return ("x".join(str(p[k]) for k in "NHWCKRS") + f"_p{p['pad_h']}{p['pad_w']}"
            f"_s{p['stride_h']}{p['stride_w']}_d{p['dil_h']}{p['dil_w']}")


# (grid width W / stride_w -> padded width)
SHAPES = [
    problem(2, 56, 56, 64, 64, 3, 3, (1, 1), (2, 2)),               # 28 -> 32
    problem(1, 6, 60, 16, 24, 3, 3, (1, 1), (2, 2)),                # 30 -> 32, one short tile
    problem(2, 20, 30, 32, 16, 3, 3, (1, 1), (2, 1)),               # stride (2, 1): 30 -> 32
    problem(1, 30, 93, 16, 24, 3, 3, (1, 1), (3, 3)),               # stride 3: 31 -> 32
    problem(2, 24, 60, 16, 16, 3, 3, (2, 2), (2, 2), (2, 2)),       # classes without taps
    problem(2, 28, 56, 128, 64, 1, 1, (0, 0), (2, 2)),              # 1x1 s2, 64-column boxes
    problem(1, 16, 128, 200, 72, 3, 3, (1, 1), (2, 2)),             # 64 -> 64, ragged C and K
    problem(1, 12, 64, 8, 8, 4, 4, (1, 1), (2, 2)),                 # even filter, 8 channels
]


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
def test_padded_rows_integer_exact(pb):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 71, cin=True)
    ref, _ = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]), want_abs=True)
    refb, _ = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]), Cin=f64(inp["C_dgrad"]),
                           alpha=0.5, beta=2.0, want_abs=True)
    out = both_settings(lambda: (run_dgrad(pb, inp, "f16"),
                                 run_dgrad(pb, inp, "f16", 0.5, 2.0)))
    for mode, (got, gotb) in out.items():
        assert_exact(got, ref, "f16", f"dgrad rows mode {mode}")
        assert_exact(gotb, refb, "f16", f"dgrad rows mode {mode}, beta")


@pytest.mark.parametrize("pb", [SHAPES[0], SHAPES[3], SHAPES[6]], ids=_id)
def test_padded_rows_random_bit_identical(pb):
    inp, P, Q = inputs(pb, "bf16", "normal_he", 73)
    ref, A = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]), want_abs=True)
    out = both_settings(lambda: run_dgrad(pb, inp, "bf16"))
    assert_close(out[0], ref, A, "bf16", "padded rows")
    np.testing.assert_array_equal(out[0], out[1])


def test_grouped_dgrad_padded_rows():
    """The block-diagonal grouped dgrad takes the same padded rows."""
    pb, G = problem(2, 28, 56, 64, 64, 3, 3, (1, 1), (2, 2)), 8
    inp, P, Q = inputs(pb, "f16", "int_uniform", 79, cin=True, groups=G)
    ref = oracle.grouped_dgrad(pb, G, f64(inp["dY"]), f64(inp["W"]))

    def run():
        dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]), torch.float16, "cuda")
        need = igc.conv2d_grouped_dgrad_workspace_size(pb, G, torch.float16)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        igc.conv2d_grouped_dgrad_ws(pb, G, torch.float16, inp["dY"].cuda(), inp["W"].cuda(),
                                    None, dX, 1.0, 0.0, ws)
        device_ok()
        check()
        return to_f64(dX)

    for mode, got in both_settings(run).items():
        assert_exact(got, ref, "f16", f"grouped dgrad rows mode {mode}")
