"""Programmatic dependent launch of the implicit-GEMM kernels and the wgrad
split reductions (IGCONV_TUNE_PDL = 1).

With the knob set, these kernels launch with the programmatic
stream-serialization attribute: the next one may start launching while the
one before it in the stream finishes, and waits (griddepcontrol.wait) for
that kernel to complete before it touches global memory.  Chains in which
every call reads the output of an earlier call, and calls that reuse one
workspace, must give bit for bit what plain launches (the built-in 0) give:
issued on one stream without synchronisation, and replayed from a CUDA
graph, where the launches become programmatic edges.  The chain's first
layer is also checked against the oracle, so the comparison is not between
two wrong answers.
"""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import assert_close, device_ok, problem, to_f64

pytestmark = pytest.mark.gpu

N, H, W = 16, 56, 56
L3 = problem(N, H, W, 64, 64, 3, 3, (1, 1))   # halo fprop / dgrad / wgrad
L1 = problem(N, H, W, 64, 64, 1, 1)           # one-issuer 1x1, split-K wgrad
L3S = problem(N, 2 * H, 2 * W, 64, 64, 3, 3, (1, 1), (2, 2))  # strided: residue classes


def data(seed):
    g = torch.Generator().manual_seed(seed)

    def rnd(*shape):
        return (torch.randn(*shape, generator=g) * 0.25).to(torch.bfloat16).cuda()
    return {"X": rnd(N, H, W, 64), "W3": rnd(64, 3, 3, 64), "W1": rnd(64, 1, 1, 64),
            "b": rnd(64), "XS": rnd(N, 2 * H, 2 * W, 64), "WS": rnd(64, 3, 3, 64)}


def chain(d):
    """Nine calls, each but the first reading the output of an earlier one."""
    Y1 = igc.fprop(L3, d["X"], d["W3"], bias=d["b"], relu=True)
    Y2 = igc.fprop(L1, Y1, d["W1"], bias=d["b"], relu=True)
    Y3 = igc.fprop(L3, Y2, d["W3"])
    dX3 = igc.dgrad(L3, Y3, d["W3"])
    dX2 = igc.dgrad(L1, dX3, d["W1"])
    dW3 = igc.wgrad(L3, Y2, Y3)
    dW1 = igc.wgrad(L1, Y1, dX3)
    dXS = igc.dgrad(L3S, dX2, d["WS"])
    dWS = igc.wgrad(L3S, dXS, dX2)
    return [Y1, Y2, Y3, dX3, dX2, dW3, dW1, dXS, dWS]


def with_pdl(mode, fn):
    try:
        igc.igconv_set_tuning(igc.TUNE_PDL, mode)
        out = fn()
        torch.cuda.synchronize()
        device_ok()
        return out
    finally:
        igc.igconv_set_tuning(igc.TUNE_PDL, 0)


def same(a, b, what):
    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), f"{what}: output {i}"


def test_chain_matches_plain_launches():
    d = data(11)
    plain = with_pdl(0, lambda: chain(d))
    for rep in range(3):
        got = with_pdl(1, lambda: chain(d))
        same(got, plain, f"stream, repetition {rep}")


def test_chain_first_layer_against_oracle():
    d = data(12)
    Y1 = with_pdl(1, lambda: chain(d))[0]
    idx = np.random.default_rng(5).choice(Y1.numel(), 8192, replace=False)
    ref, A = oracle.fprop(L3, to_f64(d["X"]), to_f64(d["W3"]), bias=to_f64(d["b"]), relu=True,
                          idx=idx, want_abs=True)
    assert_close(to_f64(Y1).reshape(-1)[idx], ref, A, "bf16", "chain layer 1")


def test_chain_in_graph_matches_plain_launches():
    d = data(13)
    plain = with_pdl(0, lambda: chain(d))

    def captured():
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            chain(d)               # warm-up outside the capture (plans, attributes)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            outs = chain(d)
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        first = [o.clone() for o in outs]
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        return first, outs

    first, last = with_pdl(1, captured)
    same(first, plain, "graph replay")
    same(last, plain, "graph, third replay")


def test_shared_workspace_back_to_back():
    """Two wgrad calls through one workspace: the second call's GEMM writes
    the partials that the first call's reduction reads."""
    da, db = data(21), data(22)
    need = max(igc.conv2d_wgrad_workspace_size(pb, torch.bfloat16, torch.bfloat16)
               for pb in (L3, L1))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def run():
        return [igc.wgrad(L3, da["X"], db["X"], workspace=ws),
                igc.wgrad(L1, db["X"], da["X"], workspace=ws),
                igc.wgrad(L3, db["X"], da["X"], workspace=ws)]

    def separate():
        out = []
        for pb, x, dy in ((L3, da["X"], db["X"]), (L1, db["X"], da["X"]),
                          (L3, db["X"], da["X"])):
            out.append(igc.wgrad(pb, x, dy))
            torch.cuda.synchronize()
        return out

    ref = with_pdl(0, separate)
    same(with_pdl(1, run), ref, "shared workspace")
    ref64 = oracle.wgrad(L1, to_f64(db["X"]), to_f64(da["X"]), want_abs=True)
    assert_close(to_f64(ref[1]), ref64[0], ref64[1], "bf16", "1x1 wgrad")
    assert np.isfinite(to_f64(ref[0])).all()
