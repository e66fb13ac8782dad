"""GPU parity of 64-wide plans with one MMA issuer per tile.

fprop and dgrad with 64-wide tiles of at most four reduction blocks (1x1
layers, the packed stem, strided dgrad's residue classes, small filters)
give each tile to one of the two MMA issuers, which adds all its blocks into
one accumulator; two epilogue groups take alternate tiles and store
64-column boxes.  A stage of the ring
then serves both issuers over time (with three blocks per tile, consecutive
fills of a stage go to different issuers), so the issuer that skips a tile
still waits for each of its fills and arrives on the stage's empty barrier:
a stage is refilled only after both issuers have seen it.  IGCONV_TUNE_ONE_ISSUER = 1 keeps two issuers per
tile.  Both settings must be exact against the oracle on integer data and
repeat bit for bit on random data.
"""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import (assert_close, assert_exact, device_ok, f64, inputs, problem,
                           to_f64)

pytestmark = pytest.mark.gpu


def run(kind, pb, inp, beta=0.0):
    if kind == "fprop":
        cin = inp["C_fprop"].cuda() if beta else None
        return to_f64(igc.fprop(pb, inp["X"].cuda(), inp["W"].cuda(), bias=inp["bias"].cuda(),
                                Cin=cin, beta=beta, relu=True))
    cin = inp["C_dgrad"].cuda() if beta else None
    return to_f64(igc.dgrad(pb, inp["dY"].cuda(), inp["W"].cuda(), Cin=cin, beta=beta))


def ref(kind, pb, inp, beta=0.0, want_abs=False):
    if kind == "fprop":
        return oracle.fprop(pb, f64(inp["X"]), f64(inp["W"]), bias=f64(inp["bias"]), relu=True,
                            Cin=f64(inp["C_fprop"]) if beta else None, beta=beta,
                            want_abs=want_abs)
    return oracle.dgrad(pb, f64(inp["dY"]), f64(inp["W"]),
                        Cin=f64(inp["C_dgrad"]) if beta else None, beta=beta, want_abs=want_abs)


def both(fn):
    out = {}
    try:
        for mode in (0, 1):
            igc.igconv_set_tuning(igc.TUNE_ONE_ISSUER, mode)
            out[mode] = fn()
            device_ok()
    finally:
        igc.igconv_set_tuning(igc.TUNE_ONE_ISSUER, 0)
    return out


def _id(c):
    pb = c[1]
    return (c[0] + "_" + "x".join(str(pb[k]) for k in "NHWCKRS") +
            f"_s{pb['stride_h']}{pb['stride_w']}")


CASES = [
    ("dgrad", problem(2, 15, 13, 64, 256, 1, 1)),                  # 1x1: 4 blocks of K
    ("fprop", problem(3, 14, 15, 64, 64, 1, 1)),                   # 1x1: 1 block
    ("fprop", problem(2, 21, 23, 64, 64, 2, 2, (1, 1))),           # 4 blocks, resident filter
    ("fprop", problem(2, 19, 17, 64, 48, 1, 3, (0, 1))),           # 3 blocks: stages alternate
    ("dgrad", problem(2, 17, 18, 48, 64, 3, 1, (1, 0))),           # 3 blocks, dgrad
    ("dgrad", problem(2, 23, 21, 64, 64, 3, 3, (1, 1), (2, 2))),   # residue classes 1-4 blocks
    ("dgrad", problem(2, 28, 56, 64, 64, 3, 3, (1, 1), (2, 2))),   # classes on 5D rows
    ("fprop", problem(2, 40, 42, 3, 64, 7, 7, (3, 3), (2, 2))),    # packed stem: 4 blocks
    # 1x1 fprop with K > 64 (wider tiles, two accumulators or one issuer)
    ("fprop", problem(2, 15, 13, 64, 256, 1, 1)),                  # 1x1 64 -> 256
    ("fprop", problem(2, 9, 11, 128, 192, 1, 1)),                  # 2 blocks, K ragged by tile
    ("fprop", problem(1, 7, 9, 96, 136, 1, 1)),                    # C and K ragged
    ("fprop", problem(1, 5, 5, 16, 1096, 1, 1)),                   # bias too long to stage
]


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_one_issuer_integer_exact(case):
    kind, pb = case
    inp, P, Q = inputs(pb, "f16", "int_uniform", 109, bias=True, cin=True)
    beta = 0.0 if pb["C"] < 8 else -1.0
    out = both(lambda: (run(kind, pb, inp), run(kind, pb, inp, beta=beta)))
    want, want_b = ref(kind, pb, inp), ref(kind, pb, inp, beta=beta)
    for mode, (got, got_b) in out.items():
        assert_exact(got, want, "f16", f"{kind} one-issuer mode {mode}")
        assert_exact(got_b, want_b, "f16", f"{kind} one-issuer mode {mode}, beta {beta}")


@pytest.mark.parametrize("case", [CASES[0], CASES[3], CASES[5]], ids=_id)
def test_one_issuer_random_within_bound_and_deterministic(case):
    kind, pb = case
    inp, P, Q = inputs(pb, "bf16", "normal_he", 113, bias=True)
    want, A = ref(kind, pb, inp, want_abs=True)
    out = both(lambda: (run(kind, pb, inp), run(kind, pb, inp)))
    for mode, (first, again) in out.items():
        assert_close(first, want, A, "bf16", f"{kind} one-issuer mode {mode}")
        np.testing.assert_array_equal(first, again)
