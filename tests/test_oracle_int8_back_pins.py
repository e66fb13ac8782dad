"""Pins for the oracle's int8 data and weight gradients (int32 results).

Each check reaches the result by another route: the fp64 dgrad / wgrad
(pinned on their own in test_oracle_pins.py) on the same integers, an int64
numpy im2col product (wgrad) and col2im scatter (dgrad), exact int64 adjoint
identities with the accumulator of the int8 forward pass, and hand-computed
sums that pass 2^31, where the int32 result is the sum modulo 2^32.
"""
import numpy as np
import pytest

from tests.test_oracle_abs_pins import _col2im, _im2col, _out
from tests.test_oracle_pins import _pb

PROBLEMS = [
    _pb(2, 7, 9, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1),
    _pb(1, 11, 10, 32, 16, 3, 3, 1, 1, 2, 2, 1, 1),     # stride 2
    _pb(2, 9, 8, 16, 16, 3, 2, 2, 1, 1, 1, 2, 1),       # dilation 2 in h
    _pb(1, 10, 13, 16, 48, 5, 3, 2, 1, 3, 2, 1, 2),     # stride 3 x 2, dilation in w
]


def _draw(pb, seed):
    rng = np.random.default_rng(seed)
    P, Q = _out(pb)
    X = rng.integers(-128, 128, size=(pb["N"], pb["H"], pb["W"], pb["C"])).astype(np.int8)
    Wt = rng.integers(-128, 128, size=(pb["K"], pb["R"], pb["S"], pb["C"])).astype(np.int8)
    dY = rng.integers(-128, 128, size=(pb["N"], P, Q, pb["K"])).astype(np.int8)
    return X, Wt, dY


@pytest.mark.parametrize("pb", PROBLEMS)
def test_int8_backward_equals_fp64_passes(oracle, pb):
    X, Wt, dY = _draw(pb, 401)
    dX = oracle.dgrad_int8(pb, dY, Wt)
    dW = oracle.wgrad_int8(pb, X, dY)
    # every sum is far below 2^31 and exact in float64
    np.testing.assert_array_equal(dX.astype(np.float64), oracle.dgrad(pb, dY, Wt))
    np.testing.assert_array_equal(dW.astype(np.float64), oracle.wgrad(pb, X, dY))


@pytest.mark.parametrize("pb", PROBLEMS)
def test_int8_backward_im2col_int64(oracle, pb):
    X, Wt, dY = _draw(pb, 402)
    P, Q = _out(pb)
    col = _im2col(pb, X.astype(np.float64)).astype(np.int64).reshape(-1, pb["R"] * pb["S"] * pb["C"])
    dW = dY.astype(np.int64).reshape(-1, pb["K"]).T @ col
    np.testing.assert_array_equal(oracle.wgrad_int8(pb, X, dY).reshape(pb["K"], -1), dW)
    g = dY.astype(np.int64).reshape(-1, pb["K"]) @ Wt.astype(np.int64).reshape(pb["K"], -1)
    dX = _col2im(pb, g.reshape(pb["N"], P, Q, pb["R"], pb["S"], pb["C"]).astype(np.float64))
    np.testing.assert_array_equal(oracle.dgrad_int8(pb, dY, Wt), dX.astype(np.int64))


@pytest.mark.parametrize("pb", PROBLEMS)
def test_int8_backward_adjoint_identities_exact(oracle, pb):
    X, Wt, dY = _draw(pb, 403)
    _, acc = oracle.fprop_int8(pb, X, Wt, None, 1.0, 1.0, 1.0, relu=False, want_acc=True)
    _, dX = oracle.dgrad_int8(pb, dY, Wt, want_acc=True)
    _, dW = oracle.wgrad_int8(pb, X, dY, want_acc=True)
    lhs = int(np.sum(acc.astype(np.int64) * dY.astype(np.int64)))
    assert lhs == int(np.sum(X.astype(np.int64) * dX))
    assert lhs == int(np.sum(Wt.astype(np.int64) * dW))


def test_int8_wgrad_wraps_past_2_31(oracle):
    """131073 products of (-128) * (-128) = 16384 sum to 2^31 + 16384, whose
    int32 value is -2^31 + 16384."""
    pb = _pb(1, 3, 43691, 1, 1, 1, 1)            # 3 * 43691 = 131073 positions
    X = np.full((1, 3, 43691, 1), -128, np.int8)
    dY = np.full((1, 3, 43691, 1), -128, np.int8)
    dW, acc = oracle.wgrad_int8(pb, X, dY, want_acc=True)
    assert int(acc.reshape(-1)[0]) == 2 ** 31 + 16384
    assert int(dW.reshape(-1)[0]) == -2 ** 31 + 16384


def test_int8_dgrad_wraps_past_2_31(oracle):
    """The same sum over 131073 output channels of one input position wraps;
    with one weight of 127 instead of -128 the sum is 2^31 - 16256, just
    inside the int32 range, and is delivered unchanged."""
    K = 131073
    pb = _pb(1, 1, 1, 1, K, 1, 1)
    dY = np.full((1, 1, 1, K), -128, np.int8)
    Wt = np.full((K, 1, 1, 1), -128, np.int8)
    dX, acc = oracle.dgrad_int8(pb, dY, Wt, want_acc=True)
    assert int(acc.reshape(-1)[0]) == 2 ** 31 + 16384
    assert int(dX.reshape(-1)[0]) == -2 ** 31 + 16384
    Wt[7] = 127
    dX, acc = oracle.dgrad_int8(pb, dY, Wt, want_acc=True)
    assert int(acc.reshape(-1)[0]) == 2 ** 31 - 16256
    assert int(dX.reshape(-1)[0]) == 2 ** 31 - 16256


def test_int8_backward_sampled_indices_match_full(oracle):
    pb = PROBLEMS[1]
    X, Wt, dY = _draw(pb, 404)
    full = oracle.dgrad_int8(pb, dY, Wt)
    idx = np.array([0, 7, full.size // 2, full.size - 1])
    np.testing.assert_array_equal(oracle.dgrad_int8(pb, dY, Wt, idx=idx), full.reshape(-1)[idx])
    full = oracle.wgrad_int8(pb, X, dY)
    idx = np.array([1, full.size - 2])
    np.testing.assert_array_equal(oracle.wgrad_int8(pb, X, dY, idx=idx), full.reshape(-1)[idx])
