"""GPU parity of the grouped entry points (depthwise kernels) against the
oracle's grouped passes.

Integer-valued fp16 inputs make every fp32 sum exact, so those outputs must
equal the oracle rounded to the output format bit for bit, in all three
passes.  Random-normal bf16 inputs are held to the acceptance tolerance and
the per-element bound.  The shapes cover every compiled filter/stride
variant (3x3, 5x5 at strides 1 and 2, 7x7 at stride 1), the generic kernel
(rectangular filters, dilation, stride 3), the strided-dgrad phase kernel
with its tap tables (strides dividing 8) and without them (stride 3), its
shared-word row loop (2 or 3 column taps per phase on consecutive dY
columns: 3x3, 5x5 and 7x7 at stride 2, and 3x3 at stride 2 with dilation 2,
whose taps of a phase are also consecutive) and the per-tap loop beside it
(one tap per phase, four taps at stride 4 x 2, and two non-consecutive taps
per phase at stride 2 with column dilation 3),
channel counts below and between the 32-channel chunks, images whose row
count is not a multiple of the 8-row blocks, and ragged column tiles."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import GROUPED_SWEEP, WORKLOADS, sample_indices
from tests.helpers import (assert_close, assert_exact, device_ok, f64, guarded_empty, inputs,
                           problem, to_f64)

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def dw(N, H, W, C, R, S, pad=(0, 0), stride=(1, 1), dil=(1, 1)):
    return problem(N, H, W, C, C, R, S, pad, stride, dil)


SHAPES = [
    dw(2, 12, 20, 64, 3, 3, (1, 1)),                    # 3x3 s1, one chunk, ragged tiles
    dw(1, 19, 33, 24, 3, 3, (1, 1), (2, 2)),            # 3x3 s2, 24 channels
    dw(2, 17, 9, 72, 5, 5, (2, 2)),                     # 5x5 s1, 64 + 8 channels
    dw(1, 23, 18, 136, 5, 5, (2, 2), (2, 2)),           # 5x5 s2, three chunks
    dw(2, 15, 21, 40, 7, 7, (3, 3)),                    # 7x7 s1
    dw(1, 14, 26, 16, 3, 5, (1, 2)),                    # rectangular: generic kernel
    dw(2, 13, 16, 32, 3, 3, (2, 2), (1, 1), (2, 2)),    # dilation 2: generic kernel
    dw(1, 20, 22, 8, 3, 3, (1, 0), (3, 2)),             # stride 3 x 2: generic, phases
    dw(1, 9, 11, 64, 7, 7, (3, 3), (2, 2)),             # 7x7 s2: generic
    dw(2, 18, 21, 48, 3, 3, (1, 1), (1, 2)),            # stride 1 x 2: dgrad phases in w only
    dw(1, 21, 17, 16, 3, 3, (2, 2), (2, 2), (2, 2)),    # stride 2 + dilation 2
    dw(1, 17, 19, 24, 3, 3, (3, 3), (2, 2), (3, 3)),    # stride 2 + dilation 3: taps 2 apart
    dw(2, 11, 30, 24, 4, 2, (1, 0), (4, 2)),            # stride 4 x 2, even filter
    dw(3, 1, 1, 16, 1, 1),                              # 1x1 pixel images
    dw(1, 5, 5, 8, 5, 5),                               # P = Q = 1
]


def _id(p):
    return ("x".join(str(p[k]) for k in "NHWCRS") + f"_p{p['pad_h']}{p['pad_w']}"
            f"_s{p['stride_h']}{p['stride_w']}_d{p['dil_h']}{p['dil_w']}")


def run_fprop(pb, inp, fmt, bias=False, alpha=1.0, beta=0.0, relu=False, G=None):
    P, Q = igc.conv2d_output_size(pb)
    Y, check = guarded_empty((pb["N"], P, Q, pb["K"]), FMT[fmt], "cuda")
    igc.conv2d_grouped_fprop(pb, G or pb["C"], FMT[fmt], inp["X"].cuda(), inp["W"].cuda(),
                             inp["bias"].cuda() if bias else None,
                             inp["C_fprop"].cuda() if beta != 0.0 else None, Y, alpha, beta,
                             relu)
    device_ok()
    check()
    return to_f64(Y)


def run_dgrad(pb, inp, fmt, alpha=1.0, beta=0.0, G=None):
    dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]), FMT[fmt], "cuda")
    igc.conv2d_grouped_dgrad(pb, G or pb["C"], FMT[fmt], inp["dY"].cuda(), inp["W"].cuda(),
                             inp["C_dgrad"].cuda() if beta != 0.0 else None, dX, alpha, beta)
    device_ok()
    check()
    return to_f64(dX)


def run_wgrad(pb, inp, fmt, dw_fmt, alpha=1.0, beta=0.0, G=None):
    G = G or pb["C"]
    dW, check = guarded_empty((pb["K"], pb["R"], pb["S"], pb["C"] // G), FMT[dw_fmt], "cuda")
    need = igc.conv2d_grouped_wgrad_workspace_size(pb, G, FMT[fmt], FMT[dw_fmt])
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    igc.conv2d_grouped_wgrad(pb, G, FMT[fmt], FMT[dw_fmt], inp["X"].cuda(),
                             inp["dY"].cuda(), inp["C_wgrad"].cuda() if beta != 0.0 else None,
                             dW, alpha, beta, ws)
    device_ok()
    check()
    return to_f64(dW)


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
def test_depthwise_integer_exact(pb):
    G = pb["C"]
    inp, P, Q = inputs(pb, "f16", "int_uniform", 31, bias=True, cin=True, dw_dtype="f32",
                       groups=G)
    X, Wt, dY = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    for bias, relu, alpha, beta in [(False, False, 1.0, 0.0), (True, True, 1.0, 0.0),
                                    (True, False, 2.0, -1.0)]:
        got = run_fprop(pb, inp, "f16", bias=bias, relu=relu, alpha=alpha, beta=beta)
        ref = oracle.grouped_fprop(pb, G, X, Wt, bias=f64(inp["bias"]) if bias else None,
                                   Cin=f64(inp["C_fprop"]) if beta else None, alpha=alpha,
                                   beta=beta, relu=relu)
        assert_exact(got, ref, "f16", f"fprop bias={bias} relu={relu} beta={beta}")
    for alpha, beta in [(1.0, 0.0), (0.5, 2.0)]:
        got = run_dgrad(pb, inp, "f16", alpha, beta)
        ref = oracle.grouped_dgrad(pb, G, dY, Wt, Cin=f64(inp["C_dgrad"]) if beta else None,
                                   alpha=alpha, beta=beta)
        assert_exact(got, ref, "f16", f"dgrad beta={beta}")
        got = run_wgrad(pb, inp, "f16", "f32", alpha, beta)
        ref = oracle.grouped_wgrad(pb, G, X, dY, Cin=f64(inp["C_wgrad"]) if beta else None,
                                   alpha=alpha, beta=beta)
        assert_exact(got, ref, "f32", f"wgrad beta={beta}")


@pytest.mark.parametrize("pb", [SHAPES[0], SHAPES[3], SHAPES[4], SHAPES[6]], ids=_id)
@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_depthwise_random_normal(pb, fmt):
    G = pb["C"]
    inp, P, Q = inputs(pb, fmt, "normal_he", 32, bias=True, groups=G)
    X, Wt, dY = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    got = run_fprop(pb, inp, fmt, bias=True, relu=True)
    ref, A = oracle.grouped_fprop(pb, G, X, Wt, bias=f64(inp["bias"]), relu=True, want_abs=True)
    assert_close(got, ref, A, fmt, "fprop")
    got = run_dgrad(pb, inp, fmt)
    ref, A = oracle.grouped_dgrad(pb, G, dY, Wt, want_abs=True)
    assert_close(got, ref, A, fmt, "dgrad")
    for dw_fmt in ("f32", fmt):
        got = run_wgrad(pb, inp, fmt, dw_fmt)
        ref, A = oracle.grouped_wgrad(pb, G, X, dY, want_abs=True)
        assert_close(got, ref, A, dw_fmt, f"wgrad -> {dw_fmt}")


# (problem, groups) with C == K and group widths 2..32: the grouped kernels
GROUPED = [
    (problem(2, 12, 15, 64, 64, 3, 3, (1, 1)), 32),                      # width 2
    (problem(1, 14, 17, 128, 128, 3, 3, (1, 1)), 32),                    # width 4 (ResNeXt)
    (problem(2, 11, 13, 96, 96, 3, 3, (1, 1), (2, 2)), 12),              # width 8, stride 2
    (problem(1, 10, 9, 64, 64, 3, 3, (2, 2), (1, 1), (2, 2)), 4),        # width 16, dilation 2
    (problem(1, 9, 10, 64, 64, 1, 1), 2),                                # width 32, 1x1
    (problem(1, 13, 11, 48, 48, 5, 3, (2, 1), (3, 2)), 6),               # width 8, stride 3x2
    (problem(2, 7, 8, 32, 32, 3, 3, (1, 1), (2, 2)), 16),                # width 2, stride 2
]


def _gid(c):
    pb, G = c
    return _id(pb) + f"_g{G}"


@pytest.mark.parametrize("case", GROUPED, ids=_gid)
def test_grouped_integer_exact(case):
    pb, G = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 41, bias=True, cin=True, dw_dtype="f32",
                       groups=G)
    X, Wt, dY = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    for bias, relu, alpha, beta in [(True, True, 1.0, 0.0), (True, False, 2.0, -1.0)]:
        got = run_fprop(pb, inp, "f16", bias=bias, relu=relu, alpha=alpha, beta=beta, G=G)
        ref = oracle.grouped_fprop(pb, G, X, Wt, bias=f64(inp["bias"]) if bias else None,
                                   Cin=f64(inp["C_fprop"]) if beta else None, alpha=alpha,
                                   beta=beta, relu=relu)
        assert_exact(got, ref, "f16", f"grouped fprop relu={relu} beta={beta}")
    for alpha, beta in [(1.0, 0.0), (0.5, 2.0)]:
        got = run_dgrad(pb, inp, "f16", alpha, beta, G=G)
        ref = oracle.grouped_dgrad(pb, G, dY, Wt, Cin=f64(inp["C_dgrad"]) if beta else None,
                                   alpha=alpha, beta=beta)
        assert_exact(got, ref, "f16", f"grouped dgrad beta={beta}")
        got = run_wgrad(pb, inp, "f16", "f32", alpha, beta, G=G)
        ref = oracle.grouped_wgrad(pb, G, X, dY, Cin=f64(inp["C_wgrad"]) if beta else None,
                                   alpha=alpha, beta=beta)
        assert_exact(got, ref, "f32", f"grouped wgrad beta={beta}")


@pytest.mark.parametrize("case", [GROUPED[1], GROUPED[2]], ids=_gid)
def test_grouped_random_normal(case):
    pb, G = case
    inp, P, Q = inputs(pb, "bf16", "normal_he", 42, bias=True, groups=G)
    X, Wt, dY = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    got = run_fprop(pb, inp, "bf16", bias=True, relu=True, G=G)
    ref, A = oracle.grouped_fprop(pb, G, X, Wt, bias=f64(inp["bias"]), relu=True, want_abs=True)
    assert_close(got, ref, A, "bf16", "grouped fprop")
    got = run_dgrad(pb, inp, "bf16", G=G)
    ref, A = oracle.grouped_dgrad(pb, G, dY, Wt, want_abs=True)
    assert_close(got, ref, A, "bf16", "grouped dgrad")
    got = run_wgrad(pb, inp, "bf16", "f32", G=G)
    ref, A = oracle.grouped_wgrad(pb, G, X, dY, want_abs=True)
    assert_close(got, ref, A, "f32", "grouped wgrad")


# the tensor-core path of conv2d_grouped_fprop_ws: group widths 4..64
GROUPED_GEMM = [
    (problem(2, 12, 15, 128, 128, 3, 3, (1, 1)), 32),                    # width 4
    (problem(1, 14, 17, 96, 96, 3, 3, (1, 1), (2, 2)), 12),              # width 8, ragged K tile
    (problem(2, 10, 9, 64, 64, 3, 3, (2, 2), (1, 1), (2, 2)), 4),        # width 16, dilation
    (problem(1, 9, 10, 192, 192, 1, 1), 6),                              # width 32, 1x1
    (problem(1, 13, 11, 128, 128, 5, 3, (2, 1), (3, 2)), 2),             # width 64, stride 3x2
]


def run_fprop_ws(pb, inp, fmt, G, bias=False, alpha=1.0, beta=0.0, relu=False):
    P, Q = igc.conv2d_output_size(pb)
    Y, check = guarded_empty((pb["N"], P, Q, pb["K"]), FMT[fmt], "cuda")
    need = igc.conv2d_grouped_fprop_workspace_size(pb, G, FMT[fmt])
    assert need >= pb["K"] * pb["R"] * pb["S"] * pb["C"] * 2  # the block-diagonal filter
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    igc.conv2d_grouped_fprop_ws(pb, G, FMT[fmt], inp["X"].cuda(), inp["W"].cuda(),
                                inp["bias"].cuda() if bias else None,
                                inp["C_fprop"].cuda() if beta != 0.0 else None, Y, alpha, beta,
                                relu, ws)
    device_ok()
    check()
    return to_f64(Y)


@pytest.mark.parametrize("case", GROUPED_GEMM, ids=_gid)
def test_grouped_tensor_core_fprop_integer_exact(case):
    pb, G = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 43, bias=True, cin=True, groups=G)
    X, Wt = f64(inp["X"]), f64(inp["W"])
    for bias, relu, alpha, beta in [(True, True, 1.0, 0.0), (True, False, 2.0, -1.0)]:
        got = run_fprop_ws(pb, inp, "f16", G, bias=bias, relu=relu, alpha=alpha, beta=beta)
        ref = oracle.grouped_fprop(pb, G, X, Wt, bias=f64(inp["bias"]), relu=relu,
                                   Cin=f64(inp["C_fprop"]) if beta else None, alpha=alpha,
                                   beta=beta)
        assert_exact(got, ref, "f16", f"grouped tensor-core fprop relu={relu} beta={beta}")


def run_dgrad_ws(pb, inp, fmt, G, alpha=1.0, beta=0.0):
    dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]), FMT[fmt], "cuda")
    need = igc.conv2d_grouped_dgrad_workspace_size(pb, G, FMT[fmt])
    assert need >= pb["K"] * pb["R"] * pb["S"] * pb["C"] * 2
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    igc.conv2d_grouped_dgrad_ws(pb, G, FMT[fmt], inp["dY"].cuda(), inp["W"].cuda(),
                                inp["C_dgrad"].cuda() if beta != 0.0 else None, dX, alpha, beta,
                                ws)
    device_ok()
    check()
    return to_f64(dX)


@pytest.mark.parametrize("case", GROUPED_GEMM + [
    (problem(2, 13, 14, 64, 64, 3, 3, (1, 1), (2, 2)), 8),             # width 8, stride 2
    (problem(1, 12, 12, 128, 128, 4, 4, (1, 1), (2, 2), (1, 1)), 8),   # width 16, 4x4 s2
], ids=_gid)
def test_grouped_tensor_core_dgrad_integer_exact(case):
    pb, G = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 46, cin=True, groups=G)
    for alpha, beta in [(1.0, 0.0), (0.5, 2.0)]:
        got = run_dgrad_ws(pb, inp, "f16", G, alpha, beta)
        ref = oracle.grouped_dgrad(pb, G, f64(inp["dY"]), f64(inp["W"]),
                                   Cin=f64(inp["C_dgrad"]) if beta else None, alpha=alpha,
                                   beta=beta)
        assert_exact(got, ref, "f16", f"grouped tensor-core dgrad beta={beta}")


@pytest.mark.parametrize("case", GROUPED_GEMM, ids=_gid)
def test_grouped_tensor_core_wgrad_integer_exact(case):
    """conv2d_grouped_wgrad takes the block-diagonal GEMM for widths 4..64."""
    pb, G = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 47, cin=True, dw_dtype="f32", groups=G)
    for alpha, beta, dw_fmt in [(1.0, 0.0, "f32"), (0.5, 2.0, "f32"), (1.0, 0.0, "f16")]:
        if dw_fmt == "f16" and beta:
            continue
        got = run_wgrad(pb, inp, "f16", dw_fmt, alpha, beta, G=G)
        ref = oracle.grouped_wgrad(pb, G, f64(inp["X"]), f64(inp["dY"]),
                                   Cin=f64(inp["C_wgrad"]) if beta else None, alpha=alpha,
                                   beta=beta)
        assert_exact(got, ref, dw_fmt, f"grouped tensor-core wgrad beta={beta} -> {dw_fmt}")


@pytest.mark.parametrize("case", [GROUPED_GEMM[0], GROUPED_GEMM[4]], ids=_gid)
def test_grouped_tensor_core_fprop_random_normal(case):
    pb, G = case
    inp, P, Q = inputs(pb, "bf16", "normal_he", 44, bias=True, groups=G)
    got = run_fprop_ws(pb, inp, "bf16", G, bias=True, relu=True)
    ref, A = oracle.grouped_fprop(pb, G, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]),
                                  relu=True, want_abs=True)
    assert_close(got, ref, A, "bf16", "grouped tensor-core fprop")


# (problem, groups) with C != K (and one C == K width above 64): a 64-wide
# tile holds whole groups and reduces over its window of the other side's
# channels (fprop / wgrad tiles over K, dgrad tiles over C)
GROUPED_CK = [
    (problem(2, 10, 11, 64, 128, 3, 3, (1, 1)), 16),                  # 4 -> 8 per group
    (problem(1, 12, 9, 128, 64, 3, 3, (1, 1), (2, 2)), 16),           # 8 -> 4, stride 2
    (problem(2, 9, 10, 32, 64, 3, 3, (1, 1)), 32),                    # depthwise x2 multiplier
    (problem(1, 8, 9, 64, 256, 1, 1), 2),                             # 32 -> 128: two tiles a group
    (problem(1, 9, 8, 256, 64, 3, 3, (1, 1)), 4),                     # 64 -> 16: 4-block windows
    (problem(1, 8, 8, 256, 256, 3, 3, (1, 1)), 2),                    # C == K, width 128
    (problem(1, 10, 10, 48, 96, 3, 3, (2, 2), (1, 1), (2, 2)), 6),    # ragged tiles, dilation 2
]


@pytest.mark.parametrize("case", GROUPED_CK, ids=_gid)
def test_grouped_channel_ratio_integer_exact(case):
    """fprop (bias, ReLU, alpha / beta), dgrad and wgrad of grouped layers
    with C != K on the tensor cores, bit-exact against the oracle."""
    pb, G = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 48, bias=True, cin=True, dw_dtype="f32",
                       groups=G)
    X, Wt, dY = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    for bias, relu, alpha, beta in [(True, True, 1.0, 0.0), (False, False, 2.0, -1.0)]:
        got = run_fprop_ws(pb, inp, "f16", G, bias=bias, relu=relu, alpha=alpha, beta=beta)
        ref = oracle.grouped_fprop(pb, G, X, Wt, bias=f64(inp["bias"]) if bias else None,
                                   relu=relu, Cin=f64(inp["C_fprop"]) if beta else None,
                                   alpha=alpha, beta=beta)
        assert_exact(got, ref, "f16", f"grouped C != K fprop relu={relu} beta={beta}")
    for alpha, beta in [(1.0, 0.0), (0.5, 2.0)]:
        got = run_dgrad_ws(pb, inp, "f16", G, alpha, beta)
        ref = oracle.grouped_dgrad(pb, G, dY, Wt, Cin=f64(inp["C_dgrad"]) if beta else None,
                                   alpha=alpha, beta=beta)
        assert_exact(got, ref, "f16", f"grouped C != K dgrad beta={beta}")
    for alpha, beta in [(1.0, 0.0), (0.5, 2.0)]:
        got = run_wgrad(pb, inp, "f16", "f32", alpha, beta, G=G)
        ref = oracle.grouped_wgrad(pb, G, X, dY, Cin=f64(inp["C_wgrad"]) if beta else None,
                                   alpha=alpha, beta=beta)
        assert_exact(got, ref, "f32", f"grouped C != K wgrad beta={beta}")


@pytest.mark.parametrize("case", [GROUPED_CK[0], GROUPED_CK[4]], ids=_gid)
def test_grouped_channel_ratio_random_normal(case):
    pb, G = case
    inp, P, Q = inputs(pb, "bf16", "normal_he", 49, bias=True, dw_dtype="f32", groups=G)
    X, Wt, dY = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    got = run_fprop_ws(pb, inp, "bf16", G, bias=True, relu=True)
    ref, A = oracle.grouped_fprop(pb, G, X, Wt, bias=f64(inp["bias"]), relu=True, want_abs=True)
    assert_close(got, ref, A, "bf16", "grouped C != K fprop")
    got = run_dgrad_ws(pb, inp, "bf16", G)
    ref, A = oracle.grouped_dgrad(pb, G, dY, Wt, want_abs=True)
    assert_close(got, ref, A, "bf16", "grouped C != K dgrad")
    got = run_wgrad(pb, inp, "bf16", "f32", G=G)
    ref, A = oracle.grouped_wgrad(pb, G, X, dY, want_abs=True)
    assert_close(got, ref, A, "f32", "grouped C != K wgrad")


def test_grouped_ws_falls_back_to_direct_kernels():
    """Widths without a tensor-core path (depthwise, 2) take the direct
    kernel through the _ws entry point: identical bits."""
    for pb, G in [(problem(1, 9, 11, 32, 32, 3, 3, (1, 1)), 32),
                  (problem(1, 9, 11, 32, 32, 3, 3, (1, 1)), 16)]:
        inp, P, Q = inputs(pb, "bf16", "normal_he", 45, bias=True, groups=G)
        a = run_fprop(pb, inp, "bf16", bias=True, relu=True, G=G)
        ws = torch.empty(16, dtype=torch.uint8, device="cuda")
        Y = torch.empty((pb["N"], P, Q, pb["K"]), dtype=torch.bfloat16, device="cuda")
        igc.conv2d_grouped_fprop_ws(pb, G, torch.bfloat16, inp["X"].cuda(), inp["W"].cuda(),
                                    inp["bias"].cuda(), None, Y, 1.0, 0.0, True, ws)
        device_ok()
        assert np.array_equal(a, to_f64(Y))


def test_groups_one_is_the_dense_path():
    pb = problem(2, 10, 12, 16, 24, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "bf16", "normal_he", 33, bias=True)
    X, Wt, dY = inp["X"].cuda(), inp["W"].cuda(), inp["dY"].cuda()
    b = inp["bias"].cuda()
    torch.testing.assert_close(igc.grouped_fprop(pb, 1, X, Wt, bias=b, relu=True),
                               igc.fprop(pb, X, Wt, bias=b, relu=True), rtol=0, atol=0)
    torch.testing.assert_close(igc.grouped_dgrad(pb, 1, dY, Wt), igc.dgrad(pb, dY, Wt),
                               rtol=0, atol=0)
    torch.testing.assert_close(igc.grouped_wgrad(pb, 1, X, dY, dw_dtype=torch.float32),
                               igc.wgrad(pb, X, dY, dw_dtype=torch.float32), rtol=0, atol=0)
    device_ok()


def test_uncovered_groups_are_unsupported():
    # group width 64 has no direct kernel (only the workspace entry point's
    # tensor-core path); C != K has only the tensor-core path, and only when
    # a 64-wide tile holds whole groups (24 output channels per group: no)
    pb = problem(1, 8, 8, 128, 128, 3, 3, (1, 1))
    X = torch.zeros((1, 8, 8, 128), dtype=torch.bfloat16, device="cuda")
    Wt = torch.zeros((128, 3, 3, 64), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((1, 8, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(igc.IgconvError) as e:
        igc.conv2d_grouped_fprop(pb, 2, torch.bfloat16, X, Wt, None, None, Y)
    assert e.value.status == 2
    pb = problem(1, 8, 8, 24, 48, 3, 3, (1, 1))
    assert igc.conv2d_grouped_fprop_workspace_size(pb, 2, torch.bfloat16) == 0
    X = torch.zeros((1, 8, 8, 24), dtype=torch.bfloat16, device="cuda")
    Wt = torch.zeros((48, 3, 3, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(igc.IgconvError) as e:
        igc.grouped_fprop(pb, 2, X, Wt)
    assert e.value.status == 2
    device_ok()


@pytest.mark.parametrize("name", GROUPED_SWEEP)
def test_depthwise_full_size_sampled(name):
    """The bench workloads at full size: sampled outputs of all three passes
    against the oracle, computed one by one, and repeat launches identical."""
    wl = WORKLOADS[name]
    pb, fmt, G = wl["problem"], wl["dtype"], wl["groups"]
    inp, P, Q = inputs(pb, fmt, wl["recipe"], wl["seed"], bias=wl["bias"],
                       dw_dtype=wl["dw_dtype"], groups=G)
    X, Wt, dY = inp["X"].cuda(), inp["W"].cuda(), inp["dY"].cuda()
    b = inp["bias"].cuda()
    Y = igc.grouped_fprop(pb, G, X, Wt, bias=b, relu=wl["relu"])
    dX = igc.grouped_dgrad(pb, G, dY, Wt)
    dW = igc.grouped_wgrad(pb, G, X, dY, dw_dtype=FMT[wl["dw_dtype"]])
    device_ok()
    assert torch.equal(igc.grouped_fprop(pb, G, X, Wt, bias=b, relu=wl["relu"]), Y)
    assert torch.equal(igc.grouped_dgrad(pb, G, dY, Wt), dX)
    assert torch.equal(igc.grouped_wgrad(pb, G, X, dY, dw_dtype=FMT[wl["dw_dtype"]]), dW)
    Xd, Wd, dYd = f64(inp["X"]), f64(inp["W"]), f64(inp["dY"])
    iy = sample_indices(Y.numel(), 2000, 1).numpy()
    ref, A = oracle.grouped_fprop(pb, G, Xd, Wd, bias=f64(inp["bias"]), relu=wl["relu"],
                                  idx=iy, want_abs=True)
    assert_close(to_f64(Y).reshape(-1)[iy], ref, A, fmt, f"{name} fprop")
    ix = sample_indices(dX.numel(), 2000, 2).numpy()
    ref, A = oracle.grouped_dgrad(pb, G, dYd, Wd, idx=ix, want_abs=True)
    assert_close(to_f64(dX).reshape(-1)[ix], ref, A, fmt, f"{name} dgrad")
    iw = sample_indices(dW.numel(), 300, 3).numpy()
    ref, A = oracle.grouped_wgrad(pb, G, Xd, dYd, idx=iw, want_abs=True)
    assert_close(to_f64(dW).reshape(-1)[iw], ref, A, wl["dw_dtype"], f"{name} wgrad")
