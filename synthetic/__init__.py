"""Seeded synthetic inputs for the convolution workloads.

This module holds workload descriptions and random draws only: no
convolution arithmetic.  Both the oracle-side tests and the GPU path take
their inputs from here, so the two sides see identical values.

Draws are made on the CPU with ``torch.Generator().manual_seed(seed)`` in the
logical NCHW / KCRS order and then laid out channel-last (NHWC / KRSC), as the
CUTLASS Python example "03_basic_conv2d.ipynb" does in its "General setup"
section (draw [N, C, H, W], convert to channels_last).  Its integer-valued
recipe ceil(uniform(-4.5, 3.5)) gives integers in [-4, 4], so fp32
accumulation stays exact for the small workloads.

The output extent (P, Q) is passed in by the caller; this module never
computes it.
"""
from __future__ import annotations

import math

import torch

# Workloads: problem shape, data recipe and seed.  The seed of the first one is
# the one the CUTLASS example states (torch.manual_seed(1234)); the others use
# 1234 + their position, since no page fixes them.
WORKLOADS = {
    "tiny": dict(
        problem=dict(N=2, H=8, W=8, C=8, K=16, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        dtype="f16", recipe="int_uniform", bias=True, seed=1234),
    "cutlass_notebook": dict(
        problem=dict(N=32, H=28, W=28, C=64, K=128, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=2, stride_w=2, dil_h=1, dil_w=1),
        dtype="f16", recipe="int_uniform", bias=False, seed=1235),
    # ResNet-50-shaped layers, batch 128, bf16, bias + ReLU on fprop.
    "resnet50_56x56_64to64_3x3": dict(
        problem=dict(N=128, H=56, W=56, C=64, K=64, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        dtype="bf16", recipe="normal_he", bias=True, relu=True, seed=1236),
    "resnet50_56x56_64to256_1x1": dict(
        problem=dict(N=128, H=56, W=56, C=64, K=256, R=1, S=1, pad_h=0, pad_w=0,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        dtype="bf16", recipe="normal_he", bias=True, relu=True, seed=1237),
    "resnet50_28x28_128to128_3x3": dict(
        problem=dict(N=128, H=28, W=28, C=128, K=128, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        dtype="bf16", recipe="normal_he", bias=True, relu=True, seed=1238),
    "resnet50_14x14_256to256_3x3": dict(
        problem=dict(N=128, H=14, W=14, C=256, K=256, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        dtype="bf16", recipe="normal_he", bias=True, relu=True, seed=1239),
    "resnet50_7x7_512to512_3x3": dict(
        problem=dict(N=128, H=7, W=7, C=512, K=512, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        dtype="bf16", recipe="normal_he", bias=True, relu=True, seed=1240),
    # dgrad/wgrad-heavy layers, fp16 with fp32 dW.
    "dilated_112x112_64to64_3x3_d2": dict(
        problem=dict(N=64, H=112, W=112, C=64, K=64, R=3, S=3, pad_h=2, pad_w=2,
                     stride_h=1, stride_w=1, dil_h=2, dil_w=2),
        dtype="f16", recipe="normal_w005", bias=False, dw_dtype="f32", seed=1241),
    "strided_112x112_64to64_3x3_s2": dict(
        problem=dict(N=64, H=112, W=112, C=64, K=64, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=2, stride_w=2, dil_h=1, dil_w=1),
        dtype="f16", recipe="normal_w005", bias=False, dw_dtype="f32", seed=1242),
    # The first layer of ResNet-50 (3 input channels, 7x7 stride 2): the
    # few-channel fprop path.
    "resnet50_stem_224x224_3to64_7x7_s2": dict(
        problem=dict(N=128, H=224, W=224, C=3, K=64, R=7, S=7, pad_h=3, pad_w=3,
                     stride_h=2, stride_w=2, dil_h=1, dil_w=1),
        dtype="bf16", recipe="normal_he", bias=True, relu=True, seed=1244),
    # Depthwise layers (groups = C = K, filters [C][R][S]) of MobileNetV2,
    # EfficientNet-B0 and ConvNeXt-T shapes, batch 128, bf16, fp32 dW.
    "mobilenetv2_112x112_96_3x3_s2_dw": dict(
        problem=dict(N=128, H=112, W=112, C=96, K=96, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=2, stride_w=2, dil_h=1, dil_w=1),
        groups=96, dtype="bf16", recipe="normal_he", bias=True, relu=True, dw_dtype="f32",
        seed=1245),
    "mobilenetv2_56x56_144_3x3_dw": dict(
        problem=dict(N=128, H=56, W=56, C=144, K=144, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        groups=144, dtype="bf16", recipe="normal_he", bias=True, relu=True, dw_dtype="f32",
        seed=1246),
    "efficientnet_56x56_144_5x5_s2_dw": dict(
        problem=dict(N=128, H=56, W=56, C=144, K=144, R=5, S=5, pad_h=2, pad_w=2,
                     stride_h=2, stride_w=2, dil_h=1, dil_w=1),
        groups=144, dtype="bf16", recipe="normal_he", bias=True, relu=True, dw_dtype="f32",
        seed=1247),
    "convnext_56x56_96_7x7_dw": dict(
        problem=dict(N=128, H=56, W=56, C=96, K=96, R=7, S=7, pad_h=3, pad_w=3,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        groups=96, dtype="bf16", recipe="normal_he", bias=True, relu=False, dw_dtype="f32",
        seed=1248),
    # A grouped layer of ResNeXt-50 (32x4d): 128 channels in 32 groups of 4.
    "resnext50_56x56_128_3x3_g32": dict(
        problem=dict(N=128, H=56, W=56, C=128, K=128, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        groups=32, dtype="bf16", recipe="normal_he", bias=True, relu=True, dw_dtype="f32",
        seed=1249),
    # A 3D layer of an R3D-18-style video network: 16 frames of 56x56, 64
    # channels, 3x3x3 filters, batch 8.
    "r3d_16x56x56_64to64_3x3x3": dict(
        problem3d=dict(N=8, D=16, H=56, W=56, C=64, K=64, T=3, R=3, S=3, pad_d=1, pad_h=1,
                       pad_w=1, stride_d=1, stride_h=1, stride_w=1, dil_d=1, dil_h=1, dil_w=1),
        dtype="bf16", recipe="normal_he", bias=True, relu=True, seed=1250),
    # int8 quantised fprop.
    "int8_56x56_128to128_3x3": dict(
        problem=dict(N=64, H=56, W=56, C=128, K=128, R=3, S=3, pad_h=1, pad_w=1,
                     stride_h=1, stride_w=1, dil_h=1, dil_w=1),
        dtype="i8", recipe="int8", bias=True, relu=True,
        act_scale=0.02, w_scale=0.01, out_scale=0.05, seed=1243),
}

DEPTHWISE_SWEEP = [
    "mobilenetv2_112x112_96_3x3_s2_dw",
    "mobilenetv2_56x56_144_3x3_dw",
    "efficientnet_56x56_144_5x5_s2_dw",
    "convnext_56x56_96_7x7_dw",
]

GROUPED_SWEEP = DEPTHWISE_SWEEP + ["resnext50_56x56_128_3x3_g32"]

RESNET50_SWEEP = [
    "resnet50_56x56_64to64_3x3",
    "resnet50_56x56_64to256_1x1",
    "resnet50_28x28_128to128_3x3",
    "resnet50_14x14_256to256_3x3",
    "resnet50_7x7_512to512_3x3",
]

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
                "i8": torch.int8}


def _nchw_draw_to_nhwc(t: torch.Tensor) -> torch.Tensor:
    # logical [N, C, H, W] draw, stored channel-last
    return t.permute(0, 2, 3, 1).contiguous()


def _int_uniform(shape, dtype, g):
    # ceil(uniform(-4.5, 3.5)): drawn in fp32, rounded to the storage dtype,
    # then ceil, which gives integers in [-4, 4] either way
    t = torch.empty(shape, dtype=torch.float32).uniform_(-4.5, 3.5, generator=g)
    return torch.ceil(t.to(dtype))


def _normal(shape, std, dtype, g):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dtype)


def make_inputs(problem: dict, P: int, Q: int, dtype: str, recipe: str, seed: int,
                bias: bool = False, cin: bool = False, dw_dtype: str | None = None,
                groups: int = 1):
    """Draw X [N,H,W,C], W [K,R,S,C/groups], dY [N,P,Q,K], bias [K] (optional)
    and the beta operands Cin for fprop (NPQK), dgrad (NHWC), wgrad
    (KRS(C/groups)) (optional), in that order, all on the CPU.

    recipe:
      int_uniform  ceil(U(-4.5, 3.5)) for X, W, dY, C; bias integer in [-4, 4]
      normal_he    X, dY ~ N(0, 1); W ~ N(0, 2/(C/groups*R*S)); bias, C ~ N(0, 1)
      normal_w005  X, dY ~ N(0, 1); W ~ N(0, 0.05) (variance); C ~ N(0, 1)
      int8         X ~ U{-128..127}, W ~ U{-127..127}, bias ~ U[-2^14, 2^14], then
                   dY ~ U{-128..127} (for the int8 gradients; drawn last, so the
                   forward operands are the same with or without it)
    """
    N, H, W, C, K, R, S = (problem[k] for k in "NHWCKRS")
    Cg = C // groups   # filter channels: the input channels of one group
    g = torch.Generator().manual_seed(seed)
    out = {}
    if recipe == "int8":
        out["X"] = _nchw_draw_to_nhwc(
            torch.randint(-128, 128, (N, C, H, W), generator=g, dtype=torch.int32).to(torch.int8))
        out["W"] = _nchw_draw_to_nhwc(
            torch.randint(-127, 128, (K, C, R, S), generator=g, dtype=torch.int32).to(torch.int8))
        if bias:
            out["bias"] = torch.randint(-(1 << 14), (1 << 14) + 1, (K,), generator=g,
                                        dtype=torch.int32)
        out["dY"] = _nchw_draw_to_nhwc(
            torch.randint(-128, 128, (N, K, P, Q), generator=g, dtype=torch.int32).to(torch.int8))
        return out
    td = TORCH_DTYPES[dtype]
    dwd = TORCH_DTYPES[dw_dtype] if dw_dtype else td
    if recipe == "int_uniform":
        out["X"] = _nchw_draw_to_nhwc(_int_uniform((N, C, H, W), td, g))
        out["W"] = _nchw_draw_to_nhwc(_int_uniform((K, Cg, R, S), td, g))
        out["dY"] = _nchw_draw_to_nhwc(_int_uniform((N, K, P, Q), td, g))
        if bias:
            out["bias"] = torch.randint(-4, 5, (K,), generator=g, dtype=torch.int32).to(td)
        if cin:
            out["C_fprop"] = _nchw_draw_to_nhwc(_int_uniform((N, K, P, Q), td, g))
            out["C_dgrad"] = _nchw_draw_to_nhwc(_int_uniform((N, C, H, W), td, g))
            out["C_wgrad"] = _nchw_draw_to_nhwc(_int_uniform((K, Cg, R, S), dwd, g))
        return out
    if recipe == "normal_he":
        wstd = math.sqrt(2.0 / (Cg * R * S))
    elif recipe == "normal_w005":
        wstd = math.sqrt(0.05)
    else:
        raise ValueError(f"unknown recipe {recipe}")
    out["X"] = _nchw_draw_to_nhwc(_normal((N, C, H, W), 1.0, td, g))
    out["W"] = _nchw_draw_to_nhwc(_normal((K, Cg, R, S), wstd, td, g))
    out["dY"] = _nchw_draw_to_nhwc(_normal((N, K, P, Q), 1.0, td, g))
    if bias:
        out["bias"] = _normal((K,), 1.0, td, g)
    if cin:
        out["C_fprop"] = _nchw_draw_to_nhwc(_normal((N, K, P, Q), 1.0, td, g))
        out["C_dgrad"] = _nchw_draw_to_nhwc(_normal((N, C, H, W), 1.0, td, g))
        out["C_wgrad"] = _nchw_draw_to_nhwc(_normal((K, Cg, R, S), 1.0, dwd, g))
    return out


def make_inputs3d(problem: dict, Do: int, P: int, Q: int, dtype: str, recipe: str, seed: int,
                  bias: bool = False, cin: bool = False):
    """3D draws: X [N,D,H,W,C], W [K,T,R,S,C], bias [K], dY [N,Do,P,Q,K] and
    (int_uniform) the beta operands C_fprop, C_dgrad, C_wgrad,
    drawn in the logical N C D H W / K C T R S order and laid out
    channel-last.  Recipes as make_inputs (int_uniform, normal_he with the
    fan-in C*T*R*S)."""
    N, D, H, W, C, K, T, R, S = (problem[k] for k in "NDHWCKTRS")
    g = torch.Generator().manual_seed(seed)
    td = TORCH_DTYPES[dtype]
    last = lambda t: t.permute(0, 2, 3, 4, 1).contiguous()  # noqa: E731
    out = {}
    if recipe == "int_uniform":
        out["X"] = last(_int_uniform((N, C, D, H, W), td, g))
        out["W"] = last(_int_uniform((K, C, T, R, S), td, g))
        if bias:
            out["bias"] = torch.randint(-4, 5, (K,), generator=g, dtype=torch.int32).to(td)
        out["dY"] = last(_int_uniform((N, K, Do, P, Q), td, g))
        if cin:
            out["C_fprop"] = last(_int_uniform((N, K, Do, P, Q), td, g))
            out["C_dgrad"] = last(_int_uniform((N, C, D, H, W), td, g))
            out["C_wgrad"] = last(_int_uniform((K, C, T, R, S), td, g))
        return out
    if recipe != "normal_he":
        raise ValueError(f"unknown recipe {recipe}")
    out["X"] = last(_normal((N, C, D, H, W), 1.0, td, g))
    out["W"] = last(_normal((K, C, T, R, S), math.sqrt(2.0 / (C * T * R * S)), td, g))
    if bias:
        out["bias"] = _normal((K,), 1.0, td, g)
    out["dY"] = last(_normal((N, K, Do, P, Q), 1.0, td, g))
    if cin:
        out["C_fprop"] = last(_normal((N, K, Do, P, Q), 1.0, td, g))
    return out


def sample_indices(total: int, count: int, seed: int) -> torch.Tensor:
    """A seeded sample of distinct linear indices in [0, total), always
    including the first and last element, sorted."""
    g = torch.Generator().manual_seed(seed)
    count = min(count, total)
    if count >= total:
        return torch.arange(total, dtype=torch.int64)
    pick = torch.randint(0, total, (count,), generator=g, dtype=torch.int64)
    pick = torch.cat([pick, torch.tensor([0, total - 1], dtype=torch.int64)])
    return torch.unique(pick)
