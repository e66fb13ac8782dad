"""GPU parity of the halo plans (stride-1 fprop and dgrad with one
64-channel reduction block, 64 output channels at most and 2..9 taps).

Output positions run on a grid of 32, 64 or 128 columns, and every tile
reads its input rows once (the halo) for all filter taps, the filter staying
in shared memory.  The tests compare the halo kernel with the oracle (exact
on integer-valued data, including bias, ReLU, beta * Cin and dilation), as
the one-copy-per-tap path (IGCONV_TUNE_HALO = 1) does (exact on integer
data and within the accumulation bound on random data, repeatable bit for
bit); shapes the halo plan does not take must still run the general path.
"""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import (assert_close, assert_exact, device_ok, f64, inputs, problem,
                           to_f64)

pytestmark = pytest.mark.gpu


def run(kind, pb, inp, beta=0.0):
    if kind == "fprop":
        cin = inp["C_fprop"].cuda() if beta else None
        return to_f64(igc.fprop(pb, inp["X"].cuda(), inp["W"].cuda(), bias=inp["bias"].cuda(),
                                Cin=cin, beta=beta, relu=True))
    cin = inp["C_dgrad"].cuda() if beta else None
    return to_f64(igc.dgrad(pb, inp["dY"].cuda(), inp["W"].cuda(), Cin=cin, beta=beta))


def ref(kind, pb, inp, beta=0.0, want_abs=False):
    if kind == "fprop":
        return oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True,
                            Cin=f64(inp["C_fprop"]) if beta else None, beta=beta,
                            want_abs=want_abs)
    return oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]),
                        Cin=f64(inp["C_dgrad"]) if beta else None, beta=beta, want_abs=want_abs)


def both(fn):
    out = {}
    try:
        for mode in (0, 1):
            igc.igconv_set_tuning(igc.TUNE_HALO, mode)
            out[mode] = fn()
            device_ok()
    finally:
        igc.igconv_set_tuning(igc.TUNE_HALO, 0)
    return out


def _id(c):
    pb = c[1]
    return (c[0] + "_" + "x".join(str(pb[k]) for k in "NHWCKRS") +
            f"_p{pb['pad_h']}_d{pb['dil_h']}")


# (grid width, output rows per 128-row tile)
CASES = [
    ("fprop", problem(2, 56, 56, 64, 64, 3, 3, (1, 1))),               # 64, 2
    ("dgrad", problem(2, 56, 56, 64, 64, 3, 3, (1, 1))),               # 64, 2
    ("fprop", problem(1, 28, 30, 32, 48, 3, 3, (1, 1))),               # 32, 4; C, K < 64
    ("dgrad", problem(1, 28, 30, 48, 32, 3, 3, (1, 1))),               # 32, 4
    ("fprop", problem(1, 16, 24, 40, 64, 3, 3, (2, 2), (1, 1), (2, 2))),   # dilation 2
    ("dgrad", problem(1, 16, 24, 40, 64, 3, 3, (2, 2), (1, 1), (2, 2))),
    ("fprop", problem(2, 10, 100, 64, 64, 1, 3, (0, 1))),              # 128, 1; 1x3 taps
    ("fprop", problem(1, 11, 61, 64, 16, 2, 2, (1, 1))),               # even filter, 64, 2
]


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_halo_integer_exact(case):
    kind, pb = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 97, bias=True, cin=True)
    out = both(lambda: (run(kind, pb, inp), run(kind, pb, inp, beta=-1.0)))
    want, want_b = ref(kind, pb, inp), ref(kind, pb, inp, beta=-1.0)
    for mode, (got, got_b) in out.items():
        assert_exact(got, want, "f16", f"{kind} halo mode {mode}")
        assert_exact(got_b, want_b, "f16", f"{kind} halo mode {mode}, beta")


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[4]], ids=_id)
def test_halo_random_within_bound_and_deterministic(case):
    """On random data the halo plan (one accumulator per tile, taps added in
    order) and the per-tap plan (two accumulators of alternating blocks)
    round differently; both stay within the fp32-accumulation bound and
    each repeats bit for bit."""
    kind, pb = case
    inp, P, Q = inputs(pb, "bf16", "normal_he", 101, bias=True)
    want, A = ref(kind, pb, inp, want_abs=True)
    out = both(lambda: (run(kind, pb, inp), run(kind, pb, inp)))
    for mode, (first, again) in out.items():
        assert_close(first, want, A, "bf16", f"{kind} halo mode {mode}")
        np.testing.assert_array_equal(first, again)


@pytest.mark.parametrize("case", [
    ("fprop", problem(2, 14, 14, 64, 64, 3, 3, (1, 1))),      # 14 rows: not a multiple of 4
    ("fprop", problem(1, 8, 150, 64, 64, 3, 3, (1, 1))),      # 152-pixel rows: wider than 128
    ("dgrad", problem(1, 20, 20, 64, 64, 5, 5, (2, 2))),      # 25 taps
], ids=_id)
def test_ineligible_shapes_take_the_general_path(case):
    kind, pb = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 103, bias=True)
    got = run(kind, pb, inp)
    device_ok()
    assert_exact(got, ref(kind, pb, inp), "f16", f"{kind} general path")


def test_halo_ignores_one_epilogue_group():
    """Halo plans store 64-column boxes, a whole tile row per warp, so they
    keep two epilogue groups even when IGCONV_TUNE_EPI_GROUPS asks for one."""
    kind, pb = CASES[0]
    inp, P, Q = inputs(pb, "f16", "int_uniform", 107, bias=True)
    want = ref(kind, pb, inp)
    try:
        igc.igconv_set_tuning(igc.TUNE_EPI_GROUPS, 1)
        got = run(kind, pb, inp)
        device_ok()
    finally:
        igc.igconv_set_tuning(igc.TUNE_EPI_GROUPS, 0)
    assert_exact(got, want, "f16", "halo with the one-group knob")
