"""Split-K forward and unit-stride data gradient (conv2d_fprop_ws /
conv2d_dgrad_ws with a workspace): each tile's reduction cut into 2-4
ranges on separate CTAs, fp32 partial tiles in the workspace, and an
ordered reduction that applies alpha, beta * Cin, bias, ReLU and the cast.
On integer data every fp32 partial and sum is exact, so the output equals
the oracle's bit for bit for every split count, including counts that do
not divide the reduction evenly; random data stays within the acceptance
tolerance.  The built-in plan never splits (it measured slower on every
ResNet-50 layer); at full size the 7x7 512 -> 512 layer at batch 128, whose
98 tiles fill two thirds of one wave of 152 SMs, is checked with 3 splits
forced."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import WORKLOADS, sample_indices
from tests.helpers import (assert_close, assert_exact, device_ok, f64, guarded_empty, inputs,
                           problem, to_f64)

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _with_splits(n, fn):
    try:
        igc.igconv_set_tuning(igc.TUNE_CONV_SPLITS, n)
        return fn()
    finally:
        igc.igconv_set_tuning(igc.TUNE_CONV_SPLITS, 0)


def run_fprop(pb, inp, fmt, bias=False, alpha=1.0, beta=0.0, relu=False):
    P, Q = igc.conv2d_output_size(pb)
    need = igc.conv2d_fprop_workspace_size(pb, FMT[fmt])
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    Y, check = guarded_empty((pb["N"], P, Q, pb["K"]), FMT[fmt], "cuda")
    igc.conv2d_fprop_ws(pb, FMT[fmt], inp["X"].cuda(), inp["W"].cuda(),
                        inp["bias"].cuda() if bias else None,
                        inp["C_fprop"].cuda() if beta != 0.0 else None, Y, alpha, beta, relu,
                        workspace=ws)
    device_ok()
    check()
    return to_f64(Y), need


def run_dgrad(pb, inp, fmt, alpha=1.0, beta=0.0):
    need = igc.conv2d_dgrad_workspace_size(pb, FMT[fmt])
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]), FMT[fmt], "cuda")
    igc.conv2d_dgrad_ws(pb, FMT[fmt], inp["dY"].cuda(), inp["W"].cuda(),
                        inp["C_dgrad"].cuda() if beta != 0.0 else None, dX, alpha, beta,
                        workspace=ws)
    device_ok()
    check()
    return to_f64(dX), need


SHAPES = [
    problem(2, 9, 9, 64, 256, 3, 3, (1, 1)),          # 9 blocks: splits 2, 3, 4 uneven
    problem(3, 7, 7, 128, 72, 3, 3, (1, 1)),          # 18 blocks, ragged output tile
    problem(1, 12, 10, 96, 64, 3, 3, (2, 1), (1, 1), (2, 1)),  # dilation, ragged channels
]


def _id(p):
    return "x".join(str(p[k]) for k in "NHWCKRS") + f"_d{p['dil_h']}"


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
@pytest.mark.parametrize("splits", [2, 3, 4])
def test_splitk_fprop_exact(pb, splits):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 111, bias=True, cin=True)
    X, Wt = f64(inp["X"]), f64(inp["W"])
    for kw in (dict(), dict(bias=True, relu=True), dict(bias=True, alpha=2.0, beta=-1.0)):
        got, need = _with_splits(splits, lambda: run_fprop(pb, inp, "f16", **kw))
        assert need > 0
        ref = oracle.fprop(pb, X, Wt, bias=f64(inp["bias"]) if kw.get("bias") else None,
                           Cin=f64(inp["C_fprop"]) if kw.get("beta") else None,
                           alpha=kw.get("alpha", 1.0), beta=kw.get("beta", 0.0),
                           relu=kw.get("relu", False))
        assert_exact(got, ref, "f16", f"fprop splits={splits} {sorted(kw)}")


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
@pytest.mark.parametrize("splits", [2, 3])
def test_splitk_dgrad_exact(pb, splits):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 113, cin=True)
    for alpha, beta in ((1.0, 0.0), (0.5, 2.0)):
        got, need = _with_splits(splits, lambda: run_dgrad(pb, inp, "f16", alpha, beta))
        assert need > 0
        ref = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]),
                           Cin=f64(inp["C_dgrad"]) if beta else None, alpha=alpha, beta=beta)
        assert_exact(got, ref, "f16", f"dgrad splits={splits} beta={beta}")


@pytest.mark.parametrize("splits", [2, 4])
def test_splitk_random_within_tolerance(splits):
    pb = SHAPES[1]
    inp, P, Q = inputs(pb, "bf16", "normal_he", 117, bias=True)
    got, _ = _with_splits(splits, lambda: run_fprop(pb, inp, "bf16", bias=True, relu=True))
    ref, A = oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True,
                          want_abs=True)
    assert_close(got, ref, A, "bf16", f"fprop splits={splits}")
    got, _ = _with_splits(splits, lambda: run_dgrad(pb, inp, "bf16"))
    ref, A = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]), want_abs=True)
    assert_close(got, ref, A, "bf16", f"dgrad splits={splits}")


def test_splitk_strided_dgrad_needs_no_workspace():
    pb = problem(2, 9, 9, 64, 64, 3, 3, (1, 1), (2, 2))
    assert igc.conv2d_dgrad_workspace_size(pb, torch.float16) == 0
    inp, P, Q = inputs(pb, "f16", "int_uniform", 119)
    got, _ = _with_splits(3, lambda: run_dgrad(pb, inp, "f16"))
    assert_exact(got, oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"])), "f16", "strided dgrad")


def test_splitk_workspace_too_small_is_an_error():
    pb = SHAPES[0]
    inp, P, Q = inputs(pb, "f16", "int_uniform", 121)

    def call():
        need = igc.conv2d_fprop_workspace_size(pb, torch.float16)
        assert need > 0
        ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
        Y = torch.empty((pb["N"], P, Q, pb["K"]), dtype=torch.float16, device="cuda")
        with pytest.raises(igc.IgconvError):
            igc.conv2d_fprop_ws(pb, torch.float16, inp["X"].cuda(), inp["W"].cuda(), None, None,
                                Y, workspace=ws)
    _with_splits(2, call)
    device_ok()


@pytest.mark.parametrize("kind", ["fprop", "dgrad"])
def test_splitk_full_size(kind):
    """7x7 512 -> 512 at batch 128 with 3 splits forced (the built-in plan
    does not split it: its size query is 0); 256 seeded outputs against the
    oracle."""
    wl = WORKLOADS["resnet50_7x7_512to512_3x3"]
    pb = wl["problem"]
    assert igc.conv2d_fprop_workspace_size(pb, torch.bfloat16) == 0
    assert igc.conv2d_dgrad_workspace_size(pb, torch.bfloat16) == 0
    inp, P, Q = inputs(pb, "bf16", wl["recipe"], wl["seed"], bias=True)
    if kind == "fprop":
        got, need = _with_splits(3, lambda: run_fprop(pb, inp, "bf16", bias=True, relu=True))
    else:
        got, need = _with_splits(3, lambda: run_dgrad(pb, inp, "bf16"))
    assert need > 0
    got = got.reshape(-1)
    idx = sample_indices(got.size, 256, 23).numpy()
    if kind == "fprop":
        ref, A = oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True,
                              idx=idx, want_abs=True)
    else:
        ref, A = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]), idx=idx, want_abs=True)
    assert_close(got[idx], ref, A, "bf16", f"7x7 {kind} split-K")
