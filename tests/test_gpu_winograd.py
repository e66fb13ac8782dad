"""GPU parity of conv2d_fprop_winograd (F(2x2, 3x3)) against the oracle's
fprop, which computes the same sum directly.

Winograd's transforms are exact in real arithmetic, so the only differences
are roundings: V = Bt d B and U = G g Gt are rounded to the 16-bit type (unit
roundoff u = 2^-8 for bf16, 2^-11 for fp16), the sum over C of the products
runs in fp32, and M is rounded to 16 bits again before the output transform.
Written out, with v*, u* the exact transforms and S[xi] = sum_c |v*||u*|,

  |Y_gpu - Y| <= |alpha| * (3u + (C + 16) * 2^-24) * (1 + 4u) * W+  +  ulp(Y),
  W+ = |At| S |A|  (per output: the transform-domain magnitudes the output
                    transform adds up),

which the tests compute in float64 from the inputs (not from the library).
On small integers in fp16 every step is exact, so the output equals the
oracle's bit for bit.  The path's acceptance bound for random data (max
|err| <= 1e-2 * max sum |x*w|) is checked as well.
"""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import WORKLOADS, sample_indices
from tests.helpers import assert_exact, device_ok, f64, guarded_empty, inputs, problem, to_f64

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16}
UNIT = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}
FRAC = {"f16": 10, "bf16": 7}
BT = np.array([[1, 0, -1, 0], [0, 1, 1, 0], [0, -1, 1, 0], [0, 1, 0, -1]], np.float64)
G = np.array([[1, 0, 0], [0.5, 0.5, 0.5], [0.5, -0.5, 0.5], [0, 0, 1]], np.float64)
AT = np.array([[1, 1, 1, 0], [0, 1, -1, -1]], np.float64)


def run_wino(pb, fmt, X, Wt, bias=None, Cin=None, alpha=1.0, beta=0.0, relu=False):
    P, Q = igc.conv2d_output_size(pb)
    need = igc.conv2d_fprop_winograd_workspace_size(pb, FMT[fmt])
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    Y, check = guarded_empty((pb["N"], P, Q, pb["K"]), FMT[fmt], "cuda")
    igc.conv2d_fprop_winograd(pb, FMT[fmt], X.cuda(), Wt.cuda(),
                              None if bias is None else bias.cuda(),
                              None if Cin is None else Cin.cuda(), Y, alpha, beta, relu, ws)
    device_ok()
    check()
    return to_f64(Y)


def magnitude_bound(pb, X, Wt, outs):
    """W+ for the outputs `outs` (an [n, 4] array of (n, p, q, k)), from the
    exact transforms of the inputs' 16-bit values, tile by tile."""
    outs = np.asarray(outs, dtype=np.int64).reshape(-1, 4)
    ph, pw = pb["pad_h"], pb["pad_w"]
    H, W = pb["H"], pb["W"]
    Xp = np.zeros((pb["N"], H + 2 * ph + 4, W + 2 * pw + 4, pb["C"]))
    Xp[:, ph:ph + H, pw:pw + W, :] = X
    U = np.abs(np.einsum("ir,krsc,js->kijc", G, Wt, G))          # [K][4][4][C]
    tiles, inv = np.unique(np.stack([outs[:, 0], outs[:, 1] // 2, outs[:, 2] // 2], 1), axis=0,
                           return_inverse=True)
    inv = inv.reshape(-1)
    d = np.stack([Xp[n, 2 * ti:2 * ti + 4, 2 * tj:2 * tj + 4, :] for n, ti, tj in tiles])
    V = np.abs(np.einsum("ia,tabc,jb->tijc", BT, d, BT))         # [T][4][4][C]
    S = np.einsum("tijc,kijc->tkij", V, U)                        # [T][K][4][4]
    Sk = S[inv, outs[:, 3]]                                       # [n][4][4]
    a = outs[:, 1] - 2 * tiles[inv, 1]
    b = outs[:, 2] - 2 * tiles[inv, 2]
    return np.einsum("ni,nij,nj->n", np.abs(AT)[a], Sk, np.abs(AT)[b])


def ulp(x, fmt):
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -14 if fmt == "f16" else -126)
    return np.ldexp(1.0, (e - FRAC[fmt]).astype(np.int64))


def check_bound(got, ref, bound_w, fmt, C, alpha, what):
    u = UNIT[fmt]
    tol = abs(alpha) * (3 * u + (C + 16) * 2.0 ** -24) * (1 + 4 * u) * bound_w + ulp(ref, fmt)
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs exceed the rounding bound; "
                           f"worst ratio {float((err / tol).max()):.3f}")
    return float((err / tol).max())


SHAPES = [
    problem(2, 8, 8, 8, 16, 3, 3, (1, 1)),
    problem(2, 13, 11, 48, 64, 3, 3, (1, 1)),      # odd output extent: partial tiles
    problem(1, 9, 10, 24, 40, 3, 3, (0, 0)),       # no padding, ragged channel blocks
    problem(3, 7, 16, 128, 96, 3, 3, (2, 1)),      # pad 2 in h: P = H + 2, two blocks
    problem(2, 10, 12, 64, 256, 3, 3, (1, 1)),     # 256 output channels
]


def _id(p):
    return "x".join(str(p[k]) for k in "NHWCKRS") + f"_p{p['pad_h']}{p['pad_w']}"


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
def test_winograd_integer_exact_f16(pb):
    """Inputs in {-1, 0, 1}: V is an integer up to 4, U a multiple of 1/4 up
    to 9/4, so every M = sum_c V U is a multiple of 1/4 of magnitude at most
    9 C; with C <= 56 that is at most 504, which fp16's 11 significant bits
    hold exactly, and the output transform and epilogue are exact in fp32."""
    g = torch.Generator().manual_seed(71)
    P, Q = igc.conv2d_output_size(pb)
    X = torch.randint(-1, 2, (pb["N"], pb["H"], pb["W"], pb["C"]), generator=g).to(torch.float16)
    Wt = torch.randint(-1, 2, (pb["K"], 3, 3, pb["C"]), generator=g).to(torch.float16)
    bias = torch.randint(-4, 5, (pb["K"],), generator=g).to(torch.float16)
    Cin = torch.randint(-4, 5, (pb["N"], P, Q, pb["K"]), generator=g).to(torch.float16)
    if 9 * pb["C"] > 512:
        pytest.skip("M could leave the range fp16 holds exactly")
    for kw in (dict(), dict(bias=bias, relu=True), dict(bias=bias, Cin=Cin, alpha=2.0, beta=-1.0)):
        got = run_wino(pb, "f16", X, Wt, **kw)
        ref = oracle.fprop(pb, f64(X), f64(Wt), bias=f64(kw.get("bias")), Cin=f64(kw.get("Cin")),
                           alpha=kw.get("alpha", 1.0), beta=kw.get("beta", 0.0),
                           relu=kw.get("relu", False))
        assert_exact(got, ref, "f16", f"winograd integer {sorted(kw)}")


@pytest.mark.parametrize("pb", SHAPES, ids=_id)
@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_winograd_random_within_rounding_bound(pb, fmt):
    inp, P, Q = inputs(pb, fmt, "normal_he", 83, bias=True)
    X, Wt, bias = f64(inp["X"]), f64(inp["W"]), f64(inp["bias"])
    got = run_wino(pb, fmt, inp["X"], inp["W"], bias=inp["bias"], relu=True, alpha=0.75)
    ref, A = oracle.fprop(pb, X, Wt, bias=bias, relu=True, alpha=0.75, want_abs=True)
    outs = np.stack(np.unravel_index(np.arange(ref.size), ref.shape), 1)
    W = magnitude_bound(pb, X, Wt, outs).reshape(ref.shape)
    check_bound(got, ref, W, fmt, pb["C"], 0.75, f"winograd {fmt}")
    # the acceptance bound for random data on the same outputs
    assert float(np.abs(got - ref).max()) <= 1e-2 * float(A.max())


def test_winograd_full_size_sampled():
    """The 56x56 64->64 3x3 layer of the ResNet-50 sweep (batch 128, bf16,
    bias + ReLU) through the Winograd path: 256 seeded outputs against the
    oracle with the rounding bound."""
    wl = WORKLOADS["resnet50_56x56_64to64_3x3"]
    pb = wl["problem"]
    inp, P, Q = inputs(pb, "bf16", wl["recipe"], wl["seed"], bias=True)
    got = run_wino(pb, "bf16", inp["X"], inp["W"], bias=inp["bias"], relu=True).reshape(-1)
    idx = sample_indices(got.size, 256, 17).numpy()
    X, Wt = f64(inp["X"]), f64(inp["W"])
    ref, A = oracle.fprop(pb, X, Wt, bias=f64(inp["bias"]), relu=True, idx=idx, want_abs=True)
    outs = np.stack(np.unravel_index(idx, (pb["N"], P, Q, pb["K"])), 1)
    W = magnitude_bound(pb, X, Wt, outs)
    check_bound(got[idx], ref, W, "bf16", pb["C"], 1.0, "winograd full size")


def test_winograd_rejects_other_shapes():
    for pb in (problem(1, 8, 8, 16, 16, 3, 3, (1, 1), (2, 2)),     # stride 2
               problem(1, 8, 8, 16, 16, 5, 5, (2, 2)),             # 5x5
               problem(1, 8, 8, 16, 16, 3, 3, (2, 2), (1, 1), (2, 2))):  # dilation
        assert igc.conv2d_fprop_winograd_workspace_size(pb, torch.bfloat16) == 0
        X = torch.zeros(1, 8, 8, 16, dtype=torch.bfloat16, device="cuda")
        Wt = torch.zeros(16, pb["R"], pb["S"], 16, dtype=torch.bfloat16, device="cuda")
        P, Q = igc.conv2d_output_size(pb)
        Y = torch.zeros(1, P, Q, 16, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
        with pytest.raises(igc.IgconvError):
            igc.conv2d_fprop_winograd(pb, torch.bfloat16, X, Wt, None, None, Y, workspace=ws)
    device_ok()
