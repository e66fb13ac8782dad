"""GPU parity of conv2d_wgrad (split-K over N*P*Q plus the deterministic
reduction) against the oracle."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import WORKLOADS
from tests.helpers import (assert_close, assert_exact, device_ok, f64, guarded_empty, inputs,
                           problem, to_f64)

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def run_wgrad(pb, inp, dtype, dw_dtype, alpha=1.0, beta=0.0):
    X, dY = inp["X"].cuda(), inp["dY"].cuda()
    Cin = inp["C_wgrad"].cuda() if beta != 0.0 else None
    need = igc.conv2d_wgrad_workspace_size(pb, FMT[dtype], FMT[dw_dtype])
    ws, check_ws = guarded_empty((max(need, 16),), torch.uint8, "cuda", guard=256, fill=77)
    dW, check = guarded_empty((pb["K"], pb["R"], pb["S"], pb["C"]), FMT[dw_dtype], "cuda")
    igc.conv2d_wgrad(pb, FMT[dtype], FMT[dw_dtype], X, dY, Cin, dW, alpha, beta, ws, need)
    device_ok()
    check()
    check_ws()
    return to_f64(dW)


def oracle_wgrad(pb, inp, alpha=1.0, beta=0.0):
    return oracle.wgrad(pb, f64(inp["X"]), f64(inp["dY"]),
                        Cin=f64(inp["C_wgrad"]) if beta != 0.0 else None, alpha=alpha, beta=beta,
                        want_abs=True)


@pytest.mark.parametrize("name", ["tiny", "cutlass_notebook"])
@pytest.mark.parametrize("dw_dtype", ["f16", "f32"])
def test_page_workloads_bit_exact(name, dw_dtype):
    wl = WORKLOADS[name]
    pb = wl["problem"]
    inp, P, Q = inputs(pb, wl["dtype"], wl["recipe"], wl["seed"], cin=True, dw_dtype=dw_dtype)
    for alpha, beta in [(1.0, 0.0), (1.0, 1.0)]:
        got = run_wgrad(pb, inp, "f16", dw_dtype, alpha, beta)
        ref, _ = oracle_wgrad(pb, inp, alpha, beta)
        assert_exact(got, ref, dw_dtype, f"{name} dW {dw_dtype} beta={beta}")


def test_split_counts_exact_on_integer_data():
    # the CUTLASS example runs wgrad with parallel split-K of 5 and serial of 3
    wl = WORKLOADS["cutlass_notebook"]
    pb = wl["problem"]
    inp, P, Q = inputs(pb, wl["dtype"], wl["recipe"], wl["seed"])
    ref, _ = oracle_wgrad(pb, inp)
    try:
        for splits in (1, 3, 5, 16, 97):
            igc.igconv_set_tuning(igc.TUNE_WGRAD_SPLITS, splits)
            got = run_wgrad(pb, inp, "f16", "f32")
            assert_exact(got, ref, "f32", f"splits={splits}")
    finally:
        igc.igconv_set_tuning(igc.TUNE_WGRAD_SPLITS, 0)


SHAPES = [
    problem(2, 8, 8, 64, 64, 1, 1),
    problem(2, 9, 11, 24, 40, 3, 3, (1, 1)),
    problem(2, 12, 12, 32, 16, 3, 3, (2, 2), (1, 1), (2, 2)),
    problem(2, 13, 12, 16, 24, 3, 3, (1, 1), (2, 2)),
    problem(1, 15, 15, 8, 8, 7, 7, (3, 3), (2, 2)),
    problem(2, 8, 8, 72, 136, 3, 3, (1, 1)),
    problem(2, 10, 10, 16, 256, 1, 1),            # K > R*S*C: the swapped orientation
    problem(3, 7, 7, 128, 192, 3, 3, (1, 1)),
]


@pytest.mark.parametrize("pb", SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS") +
                         f"_p{p['pad_h']}{p['pad_w']}_s{p['stride_h']}{p['stride_w']}"
                         f"_d{p['dil_h']}{p['dil_w']}")
def test_shapes_integer_exact(pb):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 23)
    got = run_wgrad(pb, inp, "f16", "f32")
    ref, _ = oracle_wgrad(pb, inp)
    assert_exact(got, ref, "f32", "integer wgrad")


@pytest.mark.parametrize("dtype,dw_dtype", [("f16", "f16"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("pb", [SHAPES[1], SHAPES[3], SHAPES[6]],
                         ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
def test_shapes_random_normal(pb, dtype, dw_dtype):
    inp, P, Q = inputs(pb, dtype, "normal_he", 29)
    got = run_wgrad(pb, inp, dtype, dw_dtype)
    ref, A = oracle_wgrad(pb, inp)
    assert_close(got, ref, A, dw_dtype, "normal wgrad")


def test_fixed_split_is_deterministic():
    pb = problem(4, 28, 28, 64, 64, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "bf16", "normal_he", 31)
    a = run_wgrad(pb, inp, "bf16", "f32")
    b = run_wgrad(pb, inp, "bf16", "f32")
    np.testing.assert_array_equal(a, b)


def test_workspace_too_small_is_rejected():
    """Below the smallest plan's workspace (the split-K plan's partials; the
    size query reports the halo plan's larger need where that plan applies)
    the call is refused."""
    pb = WORKLOADS["tiny"]["problem"]
    inp, P, Q = inputs(pb, "f16", "int_uniform", 1)
    try:
        igc.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 1)
        need = igc.conv2d_wgrad_workspace_size(pb, torch.float16, torch.float16)
    finally:
        igc.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 0)
    assert igc.conv2d_wgrad_workspace_size(pb, torch.float16, torch.float16) >= need
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dW = torch.empty(pb["K"], pb["R"], pb["S"], pb["C"], dtype=torch.float16, device="cuda")
    with pytest.raises(igc.IgconvError) as e:
        igc.conv2d_wgrad(pb, torch.float16, torch.float16, inp["X"].cuda(), inp["dY"].cuda(), None,
                         dW, 1.0, 0.0, ws, need - 4)
    assert e.value.status == 4
