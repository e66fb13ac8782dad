"""conv2d_wgrad_noalloc: the weight gradient for callers that cannot allocate
device memory (code under a memory manager that only hands it input and
output buffers, or code that must not call cudaMalloc on its hot path).  It
keeps the split-K partial sums in the library's fixed device array instead of
a caller workspace.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.  It calls the entry point through
the C ABI on two calls in a row with different problems, so a stale array
from the first call cannot make the second pass, and checks each result
bit for bit against conv2d_wgrad (the workspace entry point), exactly
against the oracle on integer data, and within the tolerance on random
data."""
import ctypes

import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from synthetic import WORKLOADS
from tests.helpers import assert_close, assert_exact, device_ok, f64, inputs, problem, to_f64

pytestmark = pytest.mark.gpu

FMT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
SCRATCH_BYTES = 32 << 20


def _noalloc():
    lib = igc.load()
    fn = lib.conv2d_wgrad_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(igc.Problem), ctypes.c_int, ctypes.c_int, P, P, P, P,
                   ctypes.c_float, ctypes.c_float, P]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(pb, dtype, dw_dtype, X, dY, Cin, dW, alpha, beta):
    fn = _noalloc()
    p = igc.Problem.make(pb)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.byref(p), igc._dtype_code(FMT[dtype]), igc._dtype_code(FMT[dw_dtype]),
              X.data_ptr(), dY.data_ptr(), None if Cin is None else Cin.data_ptr(),
              dW.data_ptr(), alpha, beta, stream)


CASES = [
    # (problem, dtype, dw dtype, recipe, seed, alpha, beta)
    (WORKLOADS["cutlass_notebook"]["problem"], "f16", "f32", "int_uniform", 101, 1.0, 0.0),
    (problem(4, 28, 28, 64, 128, 3, 3, (1, 1), (1, 1)), "bf16", "bf16", "normal_he", 202, 1.0,
     0.5),
]


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    for pb, dt, dwt, recipe, seed, alpha, beta in CASES:
        inp, P, Q = inputs(pb, dt, recipe, seed, cin=True, dw_dtype=dwt)
        assert igc.conv2d_wgrad_workspace_size(pb, FMT[dt], FMT[dwt]) <= SCRATCH_BYTES
        X, dY = inp["X"].cuda(), inp["dY"].cuda()
        Cin = inp["C_wgrad"].cuda() if beta != 0.0 else None
        ref = igc.wgrad(pb, X, dY, dw_dtype=FMT[dwt], Cin=Cin, alpha=alpha, beta=beta)
        dW = torch.full_like(ref, 1234.0)
        rc = _call_noalloc(pb, dt, dwt, X, dY, Cin, dW, alpha, beta)
        assert rc == 0, igc.igconv_status_string(rc)
        device_ok()
        want, A = oracle.wgrad(pb, f64(inp["X"]), f64(inp["dY"]),
                               Cin=f64(inp["C_wgrad"]) if beta != 0.0 else None, alpha=alpha,
                               beta=beta, want_abs=True)
        what = f"no-alloc wgrad {pb['N']}x{pb['H']}"
        # the same plan and kernels as the workspace entry point: the same bits
        assert torch.equal(dW.view(torch.uint8), ref.view(torch.uint8)), \
            f"{what}: differs from conv2d_wgrad"
        if recipe == "int_uniform":
            # integer data whose sums stay below 2^24: exact against the oracle
            assert_exact(to_f64(dW), want, dwt, what)
        assert_close(to_f64(dW), want, A, dwt, what)


def test_noalloc_rejects_problems_beyond_the_scratch():
    # 9 taps x 1024 channels x 1024 output channels of fp32 partials: 36 MiB
    pb = problem(1, 8, 8, 1024, 1024, 3, 3, (1, 1))
    assert igc.conv2d_wgrad_workspace_size(pb, torch.float16, torch.float16) > SCRATCH_BYTES
    X = torch.zeros(1, 8, 8, 1024, dtype=torch.float16, device="cuda")
    dY = torch.zeros(1, 8, 8, 1024, dtype=torch.float16, device="cuda")
    dW = torch.zeros(1024, 3, 3, 1024, dtype=torch.float16, device="cuda")
    rc = _call_noalloc(pb, "f16", "f16", X, dY, None, dW, 1.0, 0.0)
    assert rc == 4, igc.igconv_status_string(rc)   # IGCONV_ERR_WORKSPACE
    device_ok()
