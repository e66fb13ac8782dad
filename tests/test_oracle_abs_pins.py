"""Pins for the oracle's second output, A = |alpha| * sum |x*w| per output
element, which scales every random-data tolerance of the GPU parity tests.

Because |x*w| = |x| * |w|, A is the same convolution pass run on the
absolute values of its operands, times |alpha|.  Each check computes that
product by a route that shares nothing with the oracle's loops: an explicit
im2col (zero padding, strided and dilated slices) followed by a matrix
product for fprop and wgrad, the matching col2im scatter for dgrad, and
torch's CPU float64 convolutions (grouped and 3D).  Operands are integers of
both signs, so every sum is exact in float64 and the comparison is equality;
signed data also makes sum |x*w| differ from |sum x*w|.  alpha = -0.75 checks
that A takes |alpha|, and bias, beta * Cin and ReLU are switched on to show
that none of them enters A.
"""
import numpy as np
import pytest
import torch

from tests.test_oracle_3d_pins import PROBLEMS_3D
from tests.test_oracle_grouped_pins import GROUPED_PROBLEMS
from tests.test_oracle_pins import _ints, _pb

ALPHA = -0.75

PROBLEMS_2D = [
    _pb(2, 7, 9, 3, 5, 3, 3, 1, 1, 1, 1, 1, 1),
    _pb(1, 8, 6, 4, 3, 3, 2, 2, 0, 2, 1, 1, 2),
    _pb(2, 10, 11, 2, 4, 5, 3, 2, 1, 3, 2, 2, 1),
    _pb(1, 9, 9, 5, 6, 3, 3, 0, 0, 4, 4, 1, 1),      # stride > R: uncovered dgrad rows
]


def _out(pb):
    P = (pb["H"] + 2 * pb["pad_h"] - pb["dil_h"] * (pb["R"] - 1) - 1) // pb["stride_h"] + 1
    Q = (pb["W"] + 2 * pb["pad_w"] - pb["dil_w"] * (pb["S"] - 1) - 1) // pb["stride_w"] + 1
    return P, Q


def _im2col(pb, X):
    """col[n, p, q, r, s, c] = X[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c],
    zero outside the image."""
    N, H, W, C, R, S = (pb[k] for k in "NHWCRS")
    P, Q = _out(pb)
    ph, pw, sh, sw = pb["pad_h"], pb["pad_w"], pb["stride_h"], pb["stride_w"]
    Xp = np.zeros((N, H + 2 * ph + sh * P, W + 2 * pw + sw * Q, C))
    Xp[:, ph:ph + H, pw:pw + W, :] = X
    col = np.zeros((N, P, Q, R, S, C))
    for r in range(R):
        for s in range(S):
            h0, w0 = r * pb["dil_h"], s * pb["dil_w"]
            col[:, :, :, r, s, :] = Xp[:, h0:h0 + sh * P:sh, w0:w0 + sw * Q:sw, :]
    return col


def _col2im(pb, col):
    """The adjoint scatter: dX[n, h, w, c] += col[n, p, q, r, s, c] for the
    (p, q, r, s) that read (h, w); positions in the padding are dropped."""
    N, H, W, C, R, S = (pb[k] for k in "NHWCRS")
    P, Q = _out(pb)
    ph, pw, sh, sw = pb["pad_h"], pb["pad_w"], pb["stride_h"], pb["stride_w"]
    Xp = np.zeros((N, H + 2 * ph + sh * P, W + 2 * pw + sw * Q, C))
    for r in range(R):
        for s in range(S):
            h0, w0 = r * pb["dil_h"], s * pb["dil_w"]
            Xp[:, h0:h0 + sh * P:sh, w0:w0 + sw * Q:sw, :] += col[:, :, :, r, s, :]
    return Xp[:, ph:ph + H, pw:pw + W, :]


def _operands(pb, seed):
    rng = np.random.default_rng(seed)
    P, Q = _out(pb)
    X = _ints(rng, (pb["N"], pb["H"], pb["W"], pb["C"]))
    Wt = _ints(rng, (pb["K"], pb["R"], pb["S"], pb["C"]))
    dY = _ints(rng, (pb["N"], P, Q, pb["K"]))
    return X, Wt, dY, rng


@pytest.mark.parametrize("pb", PROBLEMS_2D)
def test_fprop_abs_sum_is_im2col_of_magnitudes(oracle, pb):
    X, Wt, dY, rng = _operands(pb, 301)
    P, Q = _out(pb)
    bias = _ints(rng, (pb["K"],))
    Cin = _ints(rng, (pb["N"], P, Q, pb["K"]))
    col = _im2col(pb, np.abs(X)).reshape(pb["N"] * P * Q, -1)
    want = abs(ALPHA) * (col @ np.abs(Wt).reshape(pb["K"], -1).T)
    Y, A = oracle.fprop(pb, X, Wt, bias=bias, Cin=Cin, alpha=ALPHA, beta=0.5, relu=True,
                        want_abs=True)
    np.testing.assert_array_equal(A.reshape(-1, pb["K"]), want)
    # the signed sum's magnitude is smaller wherever terms cancel
    Y0, _ = oracle.fprop(pb, X, Wt, alpha=ALPHA, want_abs=True)
    assert (np.abs(Y0).reshape(A.shape) < A).any()


@pytest.mark.parametrize("pb", PROBLEMS_2D)
def test_dgrad_abs_sum_is_col2im_of_magnitudes(oracle, pb):
    X, Wt, dY, rng = _operands(pb, 302)
    Cin = _ints(rng, X.shape)
    P, Q = _out(pb)
    # col[n,p,q,(r,s,c)] = sum_k |dY[n,p,q,k]| |W[k,r,s,c]|, scattered back
    col = (np.abs(dY).reshape(-1, pb["K"]) @ np.abs(Wt).reshape(pb["K"], -1))
    want = abs(ALPHA) * _col2im(pb, col.reshape(pb["N"], P, Q, pb["R"], pb["S"], pb["C"]))
    _, A = oracle.dgrad(pb, dY, Wt, Cin=Cin, alpha=ALPHA, beta=2.0, want_abs=True)
    np.testing.assert_array_equal(A, want)


@pytest.mark.parametrize("pb", PROBLEMS_2D)
def test_wgrad_abs_sum_is_im2col_of_magnitudes(oracle, pb):
    X, Wt, dY, rng = _operands(pb, 303)
    Cin = _ints(rng, Wt.shape)
    col = _im2col(pb, np.abs(X)).reshape(-1, pb["R"] * pb["S"] * pb["C"])
    want = abs(ALPHA) * (np.abs(dY).reshape(-1, pb["K"]).T @ col)
    _, A = oracle.wgrad(pb, X, dY, Cin=Cin, alpha=ALPHA, beta=-1.0, want_abs=True)
    np.testing.assert_array_equal(A.reshape(pb["K"], -1), want)


def _t(a, perm):
    return torch.from_numpy(np.ascontiguousarray(a)).permute(*perm)


@pytest.mark.parametrize("pb,groups", GROUPED_PROBLEMS)
def test_grouped_abs_sums_are_torch_convs_of_magnitudes(oracle, pb, groups):
    rng = np.random.default_rng(304)
    P, Q = _out(pb)
    X = _ints(rng, (pb["N"], pb["H"], pb["W"], pb["C"]))
    Wt = _ints(rng, (pb["K"], pb["R"], pb["S"], pb["C"] // groups))
    dY = _ints(rng, (pb["N"], P, Q, pb["K"]))
    kw = dict(stride=(pb["stride_h"], pb["stride_w"]), padding=(pb["pad_h"], pb["pad_w"]),
              dilation=(pb["dil_h"], pb["dil_w"]), groups=groups)
    aX, aW, adY = _t(np.abs(X), (0, 3, 1, 2)), _t(np.abs(Wt), (0, 3, 1, 2)), \
        _t(np.abs(dY), (0, 3, 1, 2))
    y = torch.nn.functional.conv2d(aX, aW, **kw).permute(0, 2, 3, 1).numpy()
    dx = torch.nn.grad.conv2d_input(tuple(aX.shape), aW, adY, **kw).permute(0, 2, 3, 1).numpy()
    dw = torch.nn.grad.conv2d_weight(aX, tuple(aW.shape), adY, **kw).permute(0, 2, 3, 1).numpy()
    _, A = oracle.grouped_fprop(pb, groups, X, Wt, alpha=ALPHA, relu=True, want_abs=True)
    np.testing.assert_array_equal(A, abs(ALPHA) * y)
    _, A = oracle.grouped_dgrad(pb, groups, dY, Wt, alpha=ALPHA, want_abs=True)
    np.testing.assert_array_equal(A, abs(ALPHA) * dx)
    _, A = oracle.grouped_wgrad(pb, groups, X, dY, alpha=ALPHA, want_abs=True)
    np.testing.assert_array_equal(A, abs(ALPHA) * dw)


@pytest.mark.parametrize("pb", PROBLEMS_3D)
def test_3d_abs_sums_are_torch_convs_of_magnitudes(oracle, pb):
    rng = np.random.default_rng(305)
    Do, P, Q = oracle.output_dhw(pb)
    X = _ints(rng, (pb["N"], pb["D"], pb["H"], pb["W"], pb["C"]))
    Wt = _ints(rng, (pb["K"], pb["T"], pb["R"], pb["S"], pb["C"]))
    dY = _ints(rng, (pb["N"], Do, P, Q, pb["K"]))
    kw = dict(stride=(pb["stride_d"], pb["stride_h"], pb["stride_w"]),
              padding=(pb["pad_d"], pb["pad_h"], pb["pad_w"]),
              dilation=(pb["dil_d"], pb["dil_h"], pb["dil_w"]))
    perm, back = (0, 4, 1, 2, 3), (0, 2, 3, 4, 1)
    aX, aW, adY = _t(np.abs(X), perm), _t(np.abs(Wt), perm), _t(np.abs(dY), perm)
    y = torch.nn.functional.conv3d(aX, aW, **kw).permute(*back).numpy()
    dx = torch.nn.grad.conv3d_input(tuple(aX.shape), aW, adY, **kw).permute(*back).numpy()
    dw = torch.nn.grad.conv3d_weight(aX, tuple(aW.shape), adY, **kw).permute(*back).numpy()
    _, A = oracle.fprop3d(pb, X, Wt, alpha=ALPHA, want_abs=True)
    np.testing.assert_array_equal(A, abs(ALPHA) * y)
    _, A = oracle.dgrad3d(pb, dY, Wt, alpha=ALPHA, want_abs=True)
    np.testing.assert_array_equal(A, abs(ALPHA) * dx)
    _, A = oracle.wgrad3d(pb, X, dY, alpha=ALPHA, want_abs=True)
    np.testing.assert_array_equal(A, abs(ALPHA) * dw)
