"""GPU parity of the NCHW <-> NHWC permute kernels against the oracle's
permutes: bit-exact, for every element size, aligned and ragged shapes.

2- and 4-byte elements whose two transposed extents are multiples of 8 (or
4) take the register-transpose kernel; (3, 24, 5, 8), (2, 40, 4, 6) and
(2, 12, 3, 4) give it warp tiles cut short in both directions.  Other shapes,
other element sizes and unaligned pointers take the shared-memory kernel."""
import numpy as np
import pytest
import torch

import convolution_implicit_gemm_gb300 as igc
import oracle
from tests.helpers import device_ok, guarded_empty

pytestmark = pytest.mark.gpu

SHAPES = [(2, 64, 8, 8), (3, 3, 7, 7), (1, 130, 5, 13), (4, 64, 56, 56), (1, 1, 1, 1),
          (2, 17, 64, 3), (3, 24, 5, 8), (2, 40, 4, 6), (2, 12, 3, 4), (1, 256, 14, 14)]
DTYPES = [torch.int8, torch.float16, torch.float32, torch.float64]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", DTYPES)
def test_permutes_bit_exact(shape, dtype):
    N, C, H, W = shape
    g = torch.Generator().manual_seed(hash(shape) % 1000)
    src = torch.randint(-100, 100, shape, generator=g, dtype=torch.int32).to(dtype)
    d_src = src.cuda()
    nhwc, check1 = guarded_empty((N, H, W, C), dtype, "cuda")
    igc.nchw_to_nhwc(d_src, nhwc, N, C, H, W)
    back, check2 = guarded_empty((N, C, H, W), dtype, "cuda")
    igc.nhwc_to_nchw(nhwc, back, N, C, H, W)
    device_ok()
    check1()
    check2()
    want = oracle.nchw_to_nhwc(src.numpy())
    np.testing.assert_array_equal(nhwc.cpu().numpy(), want)
    np.testing.assert_array_equal(back.cpu().numpy(), src.numpy())


def test_permute_unaligned_pointer_takes_scalar_path():
    N, C, H, W = 2, 16, 8, 8
    src = torch.arange(N * C * H * W + 1, dtype=torch.float16).cuda()
    dst = torch.zeros(N * C * H * W + 1, dtype=torch.float16).cuda()
    igc.nchw_to_nhwc(src[1:], dst[1:], N, C, H, W)
    device_ok()
    want = oracle.nchw_to_nhwc(src[1:].cpu().numpy().reshape(N, C, H, W))
    np.testing.assert_array_equal(dst[1:].cpu().numpy().reshape(N, H, W, C), want)
