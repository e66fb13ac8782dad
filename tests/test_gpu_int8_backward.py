"""GPU parity of conv2d_dgrad_int8 and conv2d_wgrad_int8 against the oracle's
int8 gradients: the whole path is integer-exact (int8 operands, fp32
accumulators that never hold more than 1024 products, int32 adds), so every
int32 output must equal the oracle's.  Shapes cover stride 1 and the strided
residue classes, dilation, channel counts that leave column tiles ragged,
reductions long enough to need several accumulators per tile and several
splits, odd products that drive an accumulator right up to 2^24, a sum that
wraps past 2^31, and the full-size 56x56 128->128 3x3 layer (sampled)."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import WORKLOADS, sample_indices
from tests.helpers import device_ok, guarded_empty, inputs, problem

pytestmark = pytest.mark.gpu


def run_dgrad(pb, dY, Wt):
    need = igc.conv2d_dgrad_int8_workspace_size(pb)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dX, check = guarded_empty((pb["N"], pb["H"], pb["W"], pb["C"]), torch.int32, "cuda")
    igc.conv2d_dgrad_int8(pb, dY.cuda(), Wt.cuda(), dX, ws)
    device_ok()
    check()
    return dX.cpu().numpy()


def run_wgrad(pb, X, dY):
    need = igc.conv2d_wgrad_int8_workspace_size(pb)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dW, check = guarded_empty((pb["K"], pb["R"], pb["S"], pb["C"]), torch.int32, "cuda")
    igc.conv2d_wgrad_int8(pb, X.cuda(), dY.cuda(), dW, ws)
    device_ok()
    check()
    return dW.cpu().numpy()


SHAPES = [
    problem(2, 8, 8, 16, 16, 3, 3, (1, 1)),
    problem(2, 14, 14, 128, 128, 3, 3, (1, 1)),              # 18 blocks: two accumulators
    problem(2, 11, 9, 32, 48, 3, 3, (1, 1), (2, 1)),         # stride 2 x 1: residue classes
    problem(1, 13, 15, 48, 32, 3, 3, (2, 2), (1, 1), (2, 2)),  # dilation 2, ragged tiles
    problem(2, 9, 9, 64, 256, 3, 3, (1, 1)),                 # dgrad: 36 blocks, 4 accumulators
    problem(1, 12, 10, 16, 32, 5, 3, (2, 1), (3, 2)),        # stride 3 x 2: uncovered rows
    problem(2, 7, 7, 64, 128, 1, 1),
]


def _id(p):
    return ("x".join(str(p[k]) for k in "NHWCKRS") +
            f"_s{p['stride_h']}{p['stride_w']}_d{p['dil_h']}{p['dil_w']}")


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
def test_int8_dgrad_exact(pb):
    inp, P, Q = inputs(pb, "i8", "int8", 61)
    got = run_dgrad(pb, inp["dY"], inp["W"])
    np.testing.assert_array_equal(got, oracle.dgrad_int8(pb, inp["dY"].numpy(), inp["W"].numpy()))


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
def test_int8_wgrad_exact(pb):
    inp, P, Q = inputs(pb, "i8", "int8", 67)
    got = run_wgrad(pb, inp["X"], inp["dY"])
    np.testing.assert_array_equal(got, oracle.wgrad_int8(pb, inp["X"].numpy(), inp["dY"].numpy()))


def test_int8_wgrad_many_splits_exact():
    """8 x 28 x 28 positions: 98 reduction blocks, more than one tile's
    accumulators hold, so the plan adds splits (int32 partials summed in
    order)."""
    pb = problem(8, 28, 28, 64, 64, 3, 3, (1, 1))
    inp, P, Q = inputs(pb, "i8", "int8", 71)
    got = run_wgrad(pb, inp["X"], inp["dY"])
    np.testing.assert_array_equal(got, oracle.wgrad_int8(pb, inp["X"].numpy(), inp["dY"].numpy()))


def test_int8_dgrad_odd_products_near_2_24_exact():
    """dY = 127 and W = +-127 with one sign per input channel: every product
    is +-16129 (odd), the centre position of a 3x3 padded layer over 128
    output channels collects 9 * 128 = 1152 of them (18,580,608 > 2^24), and
    each accumulator's share of at most 1024 products climbs to 16,516,096,
    which needs all 24 significand bits.  Then 1152 output channels into one
    position through a 1x1 filter."""
    sgn = np.where(np.arange(16) % 2 == 0, 1, -1)
    pb = problem(1, 3, 3, 16, 128, 3, 3, (1, 1))
    dY = torch.full((1, 3, 3, 128), 127, dtype=torch.int8)
    Wt = torch.from_numpy((127 * np.ones((128, 3, 3, 16)) * sgn).astype(np.int8))
    got = run_dgrad(pb, dY, Wt)
    want = oracle.dgrad_int8(pb, dY.numpy(), Wt.numpy())
    assert abs(int(want[0, 1, 1, 0])) == 1152 * 16129
    np.testing.assert_array_equal(got, want)
    pb = problem(1, 3, 3, 16, 1152, 1, 1)
    dY = torch.full((1, 3, 3, 1152), 127, dtype=torch.int8)
    Wt = torch.from_numpy((127 * np.ones((1152, 1, 1, 16)) * sgn).astype(np.int8))
    got = run_dgrad(pb, dY, Wt)
    want = oracle.dgrad_int8(pb, dY.numpy(), Wt.numpy())
    assert abs(int(want.reshape(-1)[0])) == 1152 * 16129
    np.testing.assert_array_equal(got, want)


def test_int8_wgrad_wraps_past_2_31():
    """131136 products of (-128) * (-128) sum to 2^31 + 2^20; the int32 result
    is that sum modulo 2^32."""
    pb = problem(1, 1, 131136, 16, 16, 1, 1)
    X = torch.full((1, 1, 131136, 16), -128, dtype=torch.int8)
    dY = torch.full((1, 1, 131136, 16), -128, dtype=torch.int8)
    got = run_wgrad(pb, X, dY)
    assert np.all(got == -2 ** 31 + 2 ** 20)
    np.testing.assert_array_equal(got, oracle.wgrad_int8(pb, X.numpy(), dY.numpy()))


def test_int8_backward_full_size_sampled():
    """The 64 x 56 x 56, 128 -> 128, 3x3 layer of the int8 workload, as the
    benchmark runs it: 256 seeded outputs of each pass against the oracle."""
    wl = WORKLOADS["int8_56x56_128to128_3x3"]
    pb = wl["problem"]
    inp, P, Q = inputs(pb, "i8", "int8", wl["seed"], bias=True)
    dX = run_dgrad(pb, inp["dY"], inp["W"]).reshape(-1)
    idx = sample_indices(dX.size, 256, 5).numpy()
    np.testing.assert_array_equal(
        dX[idx], oracle.dgrad_int8(pb, inp["dY"].numpy(), inp["W"].numpy(), idx=idx))
    dW = run_wgrad(pb, inp["X"], inp["dY"]).reshape(-1)
    idx = sample_indices(dW.size, 256, 6).numpy()
    np.testing.assert_array_equal(
        dW[idx], oracle.wgrad_int8(pb, inp["X"].numpy(), inp["dY"].numpy(), idx=idx))


def test_int8_backward_rejects_bad_arguments():
    pb = problem(1, 8, 8, 24, 16, 3, 3, (1, 1))   # C not a multiple of 16
    X = torch.zeros(1, 8, 8, 24, dtype=torch.int8, device="cuda")
    dY = torch.zeros(1, 8, 8, 16, dtype=torch.int8, device="cuda")
    dW = torch.zeros(16, 3, 3, 24, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(igc.IgconvError):
        igc.conv2d_wgrad_int8(pb, X, dY, dW, ws)
    pb = problem(1, 8, 8, 16, 16, 3, 3, (1, 1))
    X = torch.zeros(1, 8, 8, 16, dtype=torch.int8, device="cuda")
    dW = torch.zeros(16, 3, 3, 16, dtype=torch.int32, device="cuda")
    with pytest.raises(igc.IgconvError):
        igc.conv2d_wgrad_int8(pb, X, dY, dW, ws[:16])  # workspace too small
    device_ok()
