"""GPU parity of conv2d_wgrad on input halos (stride 1, C and K at most
128, 2..9 filter taps).

Output positions run on a grid 32, 64 or 128 columns wide in blocks of 128
positions; each block's input rows (the halo, per 64-channel plane) and dY
rows (per 64-channel chunk) are copied once for all taps; (tap, plane)
entries pair into 128-row MMA tiles whose two halves point at their rows; a
CTA computes a group of tiles over its split, and the ordered split
reduction finishes dW.  Compared with the oracle (exact on
integer-valued data, alpha / beta, fp32 and 16-bit dW), with the split-K
plan (IGCONV_TUNE_WGRAD_HALO = 1; same values on integer data, both within
the bound and repeatable on random data), and with a workspace too small for
the halo partials (the split-K plan runs instead).
"""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import (assert_close, assert_exact, device_ok, f64, guarded_empty, inputs,
                           problem, to_f64)

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def run(pb, inp, dtype, dw_dtype, alpha=1.0, beta=0.0, ws_bytes=None):
    X, dY = inp["X"].cuda(), inp["dY"].cuda()
    Cin = inp["C_wgrad"].cuda() if beta != 0.0 else None
    need = igc.conv2d_wgrad_workspace_size(pb, FMT[dtype], FMT[dw_dtype])
    if ws_bytes is not None:
        need = ws_bytes
    ws, check_ws = guarded_empty((max(need, 16),), torch.uint8, "cuda", guard=256, fill=77)
    dW, check = guarded_empty((pb["K"], pb["R"], pb["S"], pb["C"]), FMT[dw_dtype], "cuda")
    igc.conv2d_wgrad(pb, FMT[dtype], FMT[dw_dtype], X, dY, Cin, dW, alpha, beta, ws, need)
    device_ok()
    check()
    check_ws()
    return to_f64(dW)


def ref(pb, inp, alpha=1.0, beta=0.0):
    return oracle.wgrad(pb, f64(inp["X"]), f64(inp["dY"]),
                        Cin=f64(inp["C_wgrad"]) if beta != 0.0 else None, alpha=alpha, beta=beta,
                        want_abs=True)


def both(fn):
    out = {}
    try:
        for mode in (0, 1):
            igc.igconv_set_tuning(igc.TUNE_WGRAD_HALO, mode)
            out[mode] = fn()
    finally:
        igc.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 0)
    return out


def _id(pb):
    return ("x".join(str(pb[k]) for k in "NHWCKRS") + f"_p{pb['pad_h']}{pb['pad_w']}"
            f"_d{pb['dil_h']}{pb['dil_w']}")


# (grid width, output rows per block): taps 9 (one lone tap), 2, 5 (1 x 5), dilation 2
SHAPES = [
    problem(2, 56, 56, 64, 64, 3, 3, (1, 1)),                   # 64, 2
    problem(1, 28, 30, 48, 32, 3, 3, (1, 1)),                   # 32, 4; C, K < 64
    problem(1, 16, 24, 40, 64, 3, 3, (2, 2), (1, 1), (2, 2)),   # dilation 2
    problem(2, 20, 40, 16, 24, 1, 5, (0, 2)),                   # 1 x 5 taps
    problem(1, 11, 61, 64, 16, 2, 2, (1, 1)),                   # 2 x 2 taps, 64-wide grid
    problem(2, 28, 28, 128, 128, 3, 3, (1, 1)),                 # two planes, N = 128, 3 groups
    problem(1, 16, 24, 96, 80, 3, 3, (2, 2), (1, 1), (2, 2)),   # ragged planes and chunks
    problem(1, 20, 30, 128, 64, 3, 1, (1, 0)),                  # two planes, N = 64
]


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
def test_wgrad_halo_integer_exact(pb):
    inp, P, Q = inputs(pb, "f16", "int_uniform", 127, cin=True, dw_dtype="f32")
    want, _ = ref(pb, inp)
    want_b, _ = ref(pb, inp, 0.5, 2.0)
    out = both(lambda: (run(pb, inp, "f16", "f32"), run(pb, inp, "f16", "f32", 0.5, 2.0)))
    for mode, (got, got_b) in out.items():
        assert_exact(got, want, "f32", f"wgrad halo mode {mode}")
        assert_exact(got_b, want_b, "f32", f"wgrad halo mode {mode}, alpha / beta")


@pytest.mark.parametrize("dw_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("pb", [SHAPES[0], SHAPES[2], SHAPES[5]], ids=_id)
def test_wgrad_halo_random_within_bound_and_deterministic(pb, dw_dtype):
    inp, P, Q = inputs(pb, "bf16", "normal_he", 131, dw_dtype=dw_dtype)
    want, A = ref(pb, inp)
    out = both(lambda: (run(pb, inp, "bf16", dw_dtype), run(pb, inp, "bf16", dw_dtype)))
    for mode, (first, again) in out.items():
        assert_close(first, want, A, dw_dtype, f"wgrad halo mode {mode}")
        np.testing.assert_array_equal(first, again)


def test_small_workspace_takes_the_split_k_plan():
    pb = SHAPES[0]
    inp, P, Q = inputs(pb, "f16", "int_uniform", 137, dw_dtype="f32")
    want, _ = ref(pb, inp)
    try:
        igc.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 1)
        small = igc.conv2d_wgrad_workspace_size(pb, torch.float16, torch.float32)
    finally:
        igc.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 0)
    full = igc.conv2d_wgrad_workspace_size(pb, torch.float16, torch.float32)
    assert full > small  # the halo plan's partials: one tile set per split
    got = run(pb, inp, "f16", "f32", ws_bytes=small)
    assert_exact(got, want, "f32", "wgrad with the split-K plan's workspace")
