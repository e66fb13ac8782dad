"""GPU parity of conv2d_fprop_int8: the whole path is integer-exact, so the
int8 outputs must equal the oracle's element for element."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import device_ok, guarded_empty, inputs, problem

pytestmark = pytest.mark.gpu


def run_int8(pb, X, Wt, bias, sa, sw, so, relu):
    P, Q = igc.conv2d_output_size(pb)
    need = igc.conv2d_fprop_int8_workspace_size(pb)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    Y, check = guarded_empty((pb["N"], P, Q, pb["K"]), torch.int8, "cuda")
    igc.conv2d_fprop_int8(pb, X.cuda(), Wt.cuda(), None if bias is None else bias.cuda(), Y,
                          sa, sw, so, relu, ws, need)
    device_ok()
    check()
    return Y.cpu().numpy()


SHAPES = [
    problem(2, 8, 8, 16, 16, 3, 3, (1, 1)),
    problem(2, 11, 9, 32, 48, 3, 3, (1, 1), (2, 1)),
    problem(1, 14, 14, 128, 128, 3, 3, (1, 1)),     # 18 reduction blocks: two accumulators
    problem(2, 7, 7, 64, 256, 1, 1),
    problem(1, 9, 9, 48, 32, 5, 5, (2, 2), (1, 1), (1, 1)),
    problem(1, 4, 5, 32, 528, 1, 1),                # bias too long to stage in smem
]


@pytest.mark.parametrize("pb", SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
@pytest.mark.parametrize("relu", [True, False])
def test_int8_exact(pb, relu):
    inp, P, Q = inputs(pb, "i8", "int8", 37, bias=True)
    got = run_int8(pb, inp["X"], inp["W"], inp["bias"], 0.02, 0.01, 0.05, relu)
    ref = oracle.fprop_int8(pb, inp["X"].numpy(), inp["W"].numpy(), inp["bias"].numpy(),
                            0.02, 0.01, 0.05, relu=relu)
    np.testing.assert_array_equal(got, ref)


def test_int8_no_bias_and_other_scales():
    pb = SHAPES[1]
    inp, P, Q = inputs(pb, "i8", "int8", 41)
    got = run_int8(pb, inp["X"], inp["W"], None, 0.5, 0.25, 7.0, False)
    ref = oracle.fprop_int8(pb, inp["X"].numpy(), inp["W"].numpy(), None, 0.5, 0.25, 7.0,
                            relu=False)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("C,num_terms", [(128, 9 * 128), (448, 9 * 448)])
def test_int8_worst_case_accumulation_is_exact(C, num_terms):
    """Every product at its extreme (-128 * -127 or -128 * 127), so the sums
    (18.7 M and 65.5 M) exceed 2^24.  A bias of -acc + j with M = 1 makes the
    output j only if the accumulator is exact to the unit."""
    K = 16
    pb = problem(2, 3, 3, C, K, 3, 3)          # P = Q = 1: every output sees every tap
    X = torch.full((2, 3, 3, C), -128, dtype=torch.int8)
    Wt = torch.empty((K, 3, 3, C), dtype=torch.int8)
    for k in range(K):
        Wt[k] = -127 if k % 2 == 0 else 127
    acc = np.array([(1 if k % 2 == 0 else -1) * num_terms * 128 * 127 for k in range(K)],
                   dtype=np.int64)
    j = np.arange(K, dtype=np.int64) - 8
    bias = torch.from_numpy((-acc + j).astype(np.int32))
    got = run_int8(pb, X, Wt, bias, 1.0, 1.0, 1.0, False)
    np.testing.assert_array_equal(got.reshape(2, K), np.stack([j, j]).astype(np.int8))


@pytest.mark.parametrize("C", [128, 448])
@pytest.mark.parametrize("pattern", ["same_sign", "rise_then_cancel"])
def test_int8_odd_products_near_2_24_are_exact(C, pattern):
    """Products 127 * +-127 = +-16129 are odd, so every partial sum over an odd
    number of them is odd: an adder that dropped the lowest significand bit of
    a sum between 2^23 and 2^24 would show.  An accumulator collects at most
    1024 products (16 blocks of 64 channels), 1024 * 16129 = 16,516,096 <
    2^24, which needs all 24 bits of the fp32 significand.  'same_sign' drives
    every accumulator to its largest sum; 'rise_then_cancel' adds the first
    five taps with one sign and the last four with the other, so the partial
    sums climb and the exact total is small.  With M = 1 and bias = -acc + j
    the output is j only if the accumulator is exact to the unit."""
    K = 16
    pb = problem(2, 3, 3, C, K, 3, 3)          # P = Q = 1: every output sees every tap
    X = torch.full((2, 3, 3, C), 127, dtype=torch.int8)
    sgn_k = np.array([1 if k % 2 == 0 else -1 for k in range(K)], dtype=np.int64)
    if pattern == "same_sign":
        tap_sign = np.ones(9, dtype=np.int64)
    else:
        tap_sign = np.array([1] * 5 + [-1] * 4, dtype=np.int64)
    Wn = (127 * sgn_k[:, None, None] * tap_sign[None, :, None]
          * np.ones((K, 9, C), dtype=np.int64)).reshape(K, 3, 3, C)
    Wt = torch.from_numpy(Wn.astype(np.int8))
    acc = 127 * Wn.reshape(K, -1).sum(axis=1)
    assert np.all(acc % 2 == 0) and np.abs(acc).max() < 2 ** 31
    j = np.arange(K, dtype=np.int64) - 8
    bias = torch.from_numpy((-acc + j).astype(np.int32))
    got = run_int8(pb, X, Wt, bias, 1.0, 1.0, 1.0, False)
    np.testing.assert_array_equal(got.reshape(2, K), np.stack([j, j]).astype(np.int8))
    # the oracle agrees on the same inputs (its accumulation is int64)
    ref = oracle.fprop_int8(pb, X.numpy(), Wt.numpy(), bias.numpy(), 1.0, 1.0, 1.0, relu=False)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("scales", [(1.0, 0.5, 1.0), (1.0, 1.0, 8.0), (0.5, 0.25, 3.0)])
def test_int8_requant_ties_exact(scales):
    """Small integer operands and M = 1/2 or 1/8 put many products t * M
    exactly on half-integers (ties to even) and the rest near them, so the
    epilogue's exact integer path decides a large share of the outputs;
    M = 1/24 gives values off the dyadic grid.  Every output must equal the
    oracle's."""
    pb = problem(2, 9, 9, 16, 32, 3, 3, (1, 1))
    P, Q = igc.conv2d_output_size(pb)
    g = torch.Generator().manual_seed(97)
    X = torch.randint(-3, 4, (2, 9, 9, 16), generator=g, dtype=torch.int32).to(torch.int8)
    Wt = torch.randint(-3, 4, (32, 3, 3, 16), generator=g, dtype=torch.int32).to(torch.int8)
    bias = torch.randint(-40, 41, (32,), generator=g, dtype=torch.int32)
    for relu in (False, True):
        got = run_int8(pb, X, Wt, bias, *scales, relu)
        ref = oracle.fprop_int8(pb, X.numpy(), Wt.numpy(), bias.numpy(), *scales, relu=relu)
        np.testing.assert_array_equal(got, ref)


def test_int8_extreme_bias_is_exact():
    """int32 biases near the ends of the range: the bias add is exact in 64
    bits (no wrap), so outputs saturate the way the oracle's int64 sum says."""
    pb = problem(1, 6, 6, 16, 16, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "i8", "int8", 101)
    bias = torch.tensor([2 ** 31 - 1, -2 ** 31] * 8, dtype=torch.int32)
    got = run_int8(pb, inp["X"], inp["W"], bias, 0.02, 0.01, 0.05, False)
    ref = oracle.fprop_int8(pb, inp["X"].numpy(), inp["W"].numpy(), bias.numpy(), 0.02, 0.01,
                            0.05, relu=False)
    np.testing.assert_array_equal(got, ref)


# R*S*C above 4096: more reduction blocks than the TMEM accumulators of one
# tile hold exactly, so the reduction is split into ranges of at most 64
# blocks with exact int32 partial tiles, added in split order before the
# bias, ReLU and requantisation
SPLIT_SHAPES = [
    problem(1, 7, 7, 512, 64, 3, 3, (1, 1)),          # 72 blocks: 2 splits (the 7x7 layer)
    problem(2, 9, 8, 1024, 32, 3, 3, (1, 1)),         # 144 blocks: 3 splits
    problem(1, 10, 10, 256, 48, 5, 5, (2, 2), (2, 2)),  # 100 blocks, stride 2
    problem(1, 6, 7, 4112, 16, 1, 1),                 # 65 blocks, ragged channel block
]


@pytest.mark.parametrize("pb", SPLIT_SHAPES, ids=lambda p: "x".join(str(p[k]) for k in "NHWCKRS"))
@pytest.mark.parametrize("relu", [True, False])
def test_int8_split_reduction_exact(pb, relu):
    P, Q = igc.conv2d_output_size(pb)
    need = igc.conv2d_fprop_int8_workspace_size(pb)
    fp16_copies = pb["N"] * pb["H"] * pb["W"] * pb["C"] * 2 + pb["K"] * pb["R"] * pb["S"] * pb["C"] * 2
    assert need > fp16_copies  # the int32 partial tiles come on top
    inp, P, Q = inputs(pb, "i8", "int8", 53, bias=True)
    got = run_int8(pb, inp["X"], inp["W"], inp["bias"], 0.02, 0.01, 0.05, relu)
    ref = oracle.fprop_int8(pb, inp["X"].numpy(), inp["W"].numpy(), inp["bias"].numpy(),
                            0.02, 0.01, 0.05, relu=relu)
    np.testing.assert_array_equal(got, ref)


def test_int8_split_worst_case_is_exact():
    """9216 products of -128 * -127 (or * 127) per output over three splits:
    |acc| = 149.8 M, every split's partial above 2^24.  With M = 1 and bias =
    -acc + j the output is j only if partials and their sum are exact."""
    K, C = 16, 1024
    pb = problem(2, 3, 3, C, K, 3, 3)
    X = torch.full((2, 3, 3, C), -128, dtype=torch.int8)
    Wt = torch.empty((K, 3, 3, C), dtype=torch.int8)
    for k in range(K):
        Wt[k] = -127 if k % 2 == 0 else 127
    acc = np.array([(1 if k % 2 == 0 else -1) * 9 * C * 128 * 127 for k in range(K)],
                   dtype=np.int64)
    j = np.arange(K, dtype=np.int64) - 8
    bias = torch.from_numpy((-acc + j).astype(np.int32))
    got = run_int8(pb, X, Wt, bias, 1.0, 1.0, 1.0, False)
    np.testing.assert_array_equal(got.reshape(2, K), np.stack([j, j]).astype(np.int8))
