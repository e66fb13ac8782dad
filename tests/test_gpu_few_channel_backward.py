"""GPU parity of the few-channel (C < 8) data and weight gradients against the
oracle: the first layer of a CNN, whose pixels are too narrow for a 16-byte
TMA row.

dgrad has two paths.  At dilation 1 (stride_h * stride_w * C <= 64) it is
the data gradient of the stride-1 problem over the space-to-depth packed
image, one packed pixel per column, written as fp32; each X element's
gradient is then gathered from the packed element it was copied to (beta *
Cin, the cast).  Otherwise (or with IGCONV_TUNE_FEW_CHANNELS = 1) it is the
dense data gradient over the filter padded to 8 channels, written as fp32
rows of 8 channels and finished the same way.  wgrad has two paths.  At dilation 1 (stride_h * stride_w * C <= 64) the pixels are packed
by space-to-depth into a padded image whose 128-byte windows of consecutive
packed pixels form the reduction operand's rows.  Otherwise (or with
IGCONV_TUNE_FEW_CHANNELS = 1) the pixels are copied to 8-channel rows and
each 64-row operand block packs 8 filter taps x 8 channels.  Either way the
ordered split reduction maps the rows back to (tap, channel) and writes the
C real channels.
"""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import WORKLOADS, sample_indices
from tests.helpers import (assert_close, assert_exact, device_ok, f64, guarded_empty, inputs,
                           problem, to_f64)

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

SHAPES = [
    problem(2, 32, 32, 3, 64, 7, 7, (3, 3), (2, 2)),              # stem: 7x7 stride 2
    problem(1, 17, 13, 1, 16, 3, 3, (1, 1)),                       # one channel, ragged M
    problem(3, 15, 15, 5, 40, 5, 5, (4, 4), (1, 1), (2, 2)),       # dilation 2, 25 taps
    problem(2, 9, 11, 7, 136, 3, 3, (1, 1), (2, 1)),               # K past one tile
    problem(1, 6, 6, 3, 8, 1, 1),                                  # 1x1
    problem(1, 17, 16, 2, 8, 2, 2, (0, 0), (3, 3)),                # stride > R: rows nobody reads
    problem(2, 9, 9, 4, 16, 3, 3, (1, 1), (4, 4)),                 # 16 residue classes
    problem(2, 10, 10, 6, 256, 2, 2, (1, 1)),                      # 4 taps, wide K
    problem(1, 12, 14, 3, 384, 3, 3, (1, 1)),                      # 9 taps, wide K
    problem(2, 11, 10, 7, 24, 3, 5, (1, 2), (2, 3), (2, 1)),       # stride + dilation mix
    problem(2, 40, 44, 3, 64, 11, 11, (2, 2), (4, 4)),             # 11x11 stride 4
    problem(2, 32, 32, 3, 96, 4, 4, (0, 0), (4, 4)),               # 4x4 patches, stride 4
    problem(1, 19, 23, 4, 32, 9, 9, (4, 4)),                       # 9 taps along w
    problem(2, 21, 20, 7, 24, 3, 5, (1, 2), (2, 3)),               # strides 2 x 3
    problem(2, 13, 12, 5, 16, 3, 3, (3, 0), (1, 2)),               # pad 3 > R - 1
]
FEW_PATHS = {0: "packed", 1: "taps"}


@pytest.fixture(params=list(FEW_PATHS), ids=FEW_PATHS.get)
def few_mode(request):
    igc.igconv_set_tuning(igc.TUNE_FEW_CHANNELS, request.param)
    yield request.param
    igc.igconv_set_tuning(igc.TUNE_FEW_CHANNELS, 0)


def _id(p):
    return ("x".join(str(p[k]) for k in "NHWCKRS") + f"_s{p['stride_h']}{p['stride_w']}"
            f"_d{p['dil_h']}{p['dil_w']}")


def run_dgrad(pb, inp, dtype, alpha=1.0, beta=0.0):
    dY, Wt = inp["dY"].cuda(), inp["W"].cuda()
    Cin = inp["C_dgrad"].cuda() if beta != 0.0 else None
    need = igc.conv2d_dgrad_workspace_size(pb, FMT[dtype])
    assert need > 0
    ws, check_ws = guarded_empty((need,), torch.uint8, "cuda", guard=256, fill=77)
    dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]), FMT[dtype], "cuda")
    igc.conv2d_dgrad_ws(pb, FMT[dtype], dY, Wt, Cin, dX, alpha, beta, ws)
    device_ok()
    check()
    check_ws()
    return to_f64(dX)


def run_wgrad(pb, inp, dtype, dw_dtype, alpha=1.0, beta=0.0):
    X, dY = inp["X"].cuda(), inp["dY"].cuda()
    Cin = inp["C_wgrad"].cuda() if beta != 0.0 else None
    need = igc.conv2d_wgrad_workspace_size(pb, FMT[dtype], FMT[dw_dtype])
    assert need > 0
    ws, check_ws = guarded_empty((need,), torch.uint8, "cuda", guard=256, fill=77)
    dW, check = guarded_empty((pb["K"], pb["R"], pb["S"], pb["C"]), FMT[dw_dtype], "cuda")
    igc.conv2d_wgrad(pb, FMT[dtype], FMT[dw_dtype], X, dY, Cin, dW, alpha, beta, ws, need)
    device_ok()
    check()
    check_ws()
    return to_f64(dW)


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
def test_dgrad_integer_exact(pb, few_mode):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 131, cin=True)
    for alpha, beta in [(1.0, 0.0), (1.0, 2.0), (-2.0, 0.5)]:
        got = run_dgrad(pb, inp, "f16", alpha, beta)
        ref = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]),
                           Cin=f64(inp["C_dgrad"]) if beta != 0.0 else None, alpha=alpha,
                           beta=beta)
        assert_exact(got, ref, "f16", f"few-channel dgrad alpha={alpha} beta={beta}")


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
@pytest.mark.parametrize("dw_dtype", ["f32", "f16"])
def test_wgrad_integer_exact(pb, dw_dtype, few_mode):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 137, cin=True, dw_dtype=dw_dtype)
    for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
        got = run_wgrad(pb, inp, "f16", dw_dtype, alpha, beta)
        ref = oracle.wgrad(pb, f64(inp["X"]), f64(inp["dY"]),
                           Cin=f64(inp["C_wgrad"]) if beta != 0.0 else None, alpha=alpha,
                           beta=beta)
        assert_exact(got, ref, dw_dtype, f"few-channel wgrad {dw_dtype} beta={beta}")


@pytest.mark.parametrize("pb", [SHAPES[0], SHAPES[2], SHAPES[7], SHAPES[9], SHAPES[10]], ids=_id)
def test_random_normal_bf16(pb, few_mode):
    inp, P, Q = inputs(pb, "bf16", "normal_he", 139, dw_dtype="f32")
    got = run_dgrad(pb, inp, "bf16")
    ref, A = oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]), want_abs=True)
    assert_close(got, ref, A, "bf16", "normal few-channel dgrad")
    got = run_wgrad(pb, inp, "bf16", "f32")
    ref, A = oracle.wgrad(pb, f64(inp["X"]), f64(inp["dY"]), want_abs=True)
    assert_close(got, ref, A, "f32", "normal few-channel wgrad")


def test_tile_width_and_split_knobs_agree(few_mode):
    """Every forced tile width and split count gives the same integer dW."""
    pb = SHAPES[0]
    inp, P, Q = inputs(pb, "f16", "int_uniform", 149)
    ref = oracle.wgrad(pb, f64(inp["X"]), f64(inp["dY"]))
    try:
        for bn in (64, 128, 256):
            for splits in (1, 3, 16):
                igc.igconv_set_tuning(igc.TUNE_BLOCK_N, bn)
                igc.igconv_set_tuning(igc.TUNE_WGRAD_SPLITS, splits)
                got = run_wgrad(pb, inp, "f16", "f32")
                assert_exact(got, ref, "f32", f"few-channel wgrad bn={bn} splits={splits}")
    finally:
        igc.igconv_set_tuning(igc.TUNE_BLOCK_N, 0)
        igc.igconv_set_tuning(igc.TUNE_WGRAD_SPLITS, 0)


def test_unaligned_rows_accepted(few_mode):
    """Rows of C < 8 channels are never 16-byte aligned in general: X, W, dX
    and dW one element past a 16-byte boundary are accepted."""
    pb = SHAPES[0]
    inp, P, Q = inputs(pb, "f16", "int_uniform", 151)

    def shifted(t):
        buf = torch.zeros(t.numel() + 8, dtype=t.dtype, device="cuda")
        v = buf[1:1 + t.numel()]
        v.copy_(t.reshape(-1).cuda())
        return v

    X, Wt = shifted(inp["X"]), shifted(inp["W"])
    dY = inp["dY"].cuda()
    dX = shifted(torch.zeros(pb["N"] * pb["H"] * pb["W"] * pb["C"], dtype=torch.float16))
    ws = torch.empty(igc.conv2d_dgrad_workspace_size(pb, torch.float16), dtype=torch.uint8,
                     device="cuda")
    igc.conv2d_dgrad_ws(pb, torch.float16, dY, Wt, None, dX, workspace=ws)
    dW = shifted(torch.zeros(pb["K"] * pb["R"] * pb["S"] * pb["C"], dtype=torch.float16))
    need = igc.conv2d_wgrad_workspace_size(pb, torch.float16, torch.float16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    igc.conv2d_wgrad(pb, torch.float16, torch.float16, X, dY, None, dW, 1.0, 0.0, ws, need)
    device_ok()
    assert_exact(to_f64(dX), oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"])).reshape(-1), "f16",
                 "unaligned dgrad")
    assert_exact(to_f64(dW), oracle.wgrad(pb, f64(inp["X"]), f64(inp["dY"])).reshape(-1), "f16",
                 "unaligned wgrad")


def test_needs_workspace():
    pb = SHAPES[0]
    P, Q = igc.conv2d_output_size(pb)
    dY = torch.zeros(pb["N"] * P * Q * pb["K"], dtype=torch.float16, device="cuda")
    Wt = torch.zeros(pb["K"] * pb["R"] * pb["S"] * pb["C"], dtype=torch.float16, device="cuda")
    X = torch.zeros(pb["N"] * pb["H"] * pb["W"] * pb["C"], dtype=torch.float16, device="cuda")
    dX = torch.empty_like(X)
    dW = torch.empty_like(Wt)
    with pytest.raises(igc.IgconvError, match="WORKSPACE"):
        igc.conv2d_dgrad(pb, torch.float16, dY, Wt, None, dX)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(igc.IgconvError, match="WORKSPACE"):
        igc.conv2d_dgrad_ws(pb, torch.float16, dY, Wt, None, dX, workspace=small)
    with pytest.raises(igc.IgconvError, match="WORKSPACE"):
        igc.conv2d_wgrad(pb, torch.float16, torch.float16, X, dY, None, dW, 1.0, 0.0, small, 256)
    device_ok()


def test_stem_full_size_sampled():
    """The first layer of ResNet-50 (batch 128, 224x224x3 -> 112x112x64, 7x7
    stride 2, bf16, fp32 dW) through the convenience wrappers: seeded
    samples of dX and dW against the oracle."""
    wl = WORKLOADS["resnet50_stem_224x224_3to64_7x7_s2"]
    pb = wl["problem"]
    inp, P, Q = inputs(pb, "bf16", wl["recipe"], wl["seed"], dw_dtype="f32")
    dY = inp["dY"].cuda()
    dX = igc.dgrad(pb, dY, inp["W"].cuda())
    dW = igc.wgrad(pb, inp["X"].cuda(), dY, dw_dtype=torch.float32)
    device_ok()
    X64, W64, dY64 = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    idx = sample_indices(dX.numel(), 1500, 21).numpy()
    ref, A = oracle.dgrad(pb, dY64, W64, idx=idx, want_abs=True)
    assert_close(to_f64(dX.reshape(-1)[torch.from_numpy(idx).cuda()]), ref, A, "bf16",
                 "stem dgrad")
    idx = sample_indices(dW.numel(), 200, 22).numpy()
    ref, A = oracle.wgrad(pb, X64, dY64, idx=idx, want_abs=True)
    assert_close(to_f64(dW.reshape(-1)[torch.from_numpy(idx).cuda()]), ref, A, "f32",
                 "stem wgrad")
