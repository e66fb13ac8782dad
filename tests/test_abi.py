"""Host-side checks of the C ABI that need no GPU: the library builds, loads
and exports every symbol the header declares; output sizes agree with the
oracle; invalid arguments are rejected before any device work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "igconv.h")


@pytest.fixture(scope="module")
def igc():
    from convolution_implicit_gemm_gb300 import build_lib
    build_lib.build()
    import convolution_implicit_gemm_gb300 as m
    m.load()
    return m


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"IGCONV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("conv2d_output_size", "conv2d_fprop", "conv2d_dgrad", "conv2d_wgrad",
                     "conv2d_wgrad_workspace_size", "conv2d_fprop_int8",
                     "conv2d_fprop_int8_workspace_size", "nchw_to_nhwc", "nhwc_to_nchw",
                     "igconv_get_device_status", "igconv_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(igc):
    lib = ctypes.CDLL(igc.library_path())
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings(igc):
    for code, name in igc.STATUS_NAMES.items():
        assert igc.igconv_status_string(code) == name
    assert igc.igconv_status_string(99) == "IGCONV_UNKNOWN_STATUS"


def test_output_size_matches_oracle(igc, oracle):
    for H in (1, 5, 8, 28, 56, 112, 224):
        for R in (1, 3, 7):
            for pad in (0, 1, 3):
                for stride in (1, 2, 3):
                    for dil in (1, 2):
                        pb = dict(N=1, H=H, W=H + 1, C=8, K=8, R=R, S=R, pad_h=pad, pad_w=pad,
                                  stride_h=stride, stride_w=stride, dil_h=dil, dil_w=dil)
                        P, Q = oracle.output_hw(pb)
                        if P < 1 or Q < 1:
                            with pytest.raises(igc.IgconvError) as e:
                                igc.conv2d_output_size(pb)
                            assert e.value.status == 1
                        else:
                            assert igc.conv2d_output_size(pb) == (P, Q)


def _pb(**kw):
    base = dict(N=2, H=8, W=8, C=16, K=16, R=3, S=3, pad_h=1, pad_w=1,
                stride_h=1, stride_w=1, dil_h=1, dil_w=1)
    base.update(kw)
    return base


# Fake, well-aligned addresses: every case below must be rejected by host
# validation before the library touches the device.
A, B, Cp = 0x10000, 0x20000, 0x30000


@pytest.mark.parametrize("kw,status", [
    (dict(N=0), 1), (dict(C=-1), 1), (dict(pad_h=-1), 1), (dict(stride_w=0), 1),
    (dict(dil_h=0), 1), (dict(H=2, R=5, pad_h=0), 1),
    (dict(C=12), 2), (dict(K=20), 2), (dict(stride_h=9), 2), (dict(pad_w=65), 2),
    (dict(R=65, H=200, pad_h=0), 2), (dict(dil_h=64, H=400), 2),
])
def test_fprop_rejects_invalid_problems(igc, kw, status):
    lib = igc.load()
    pb = igc.Problem.make(_pb(**kw))
    rc = lib.conv2d_fprop(ctypes.byref(pb), igc.F16, A, B, None, None, Cp, 1.0, 0.0, 0, None)
    assert rc == status


def test_fprop_rejects_bad_pointers_and_scalars(igc):
    lib = igc.load()
    pb = igc.Problem.make(_pb())
    assert lib.conv2d_fprop(ctypes.byref(pb), igc.F16, None, B, None, None, Cp, 1.0, 0.0, 0, None) == 1
    assert lib.conv2d_fprop(ctypes.byref(pb), igc.F16, A, B, None, None, Cp, 1.0, 1.0, 0, None) == 1
    assert lib.conv2d_fprop(ctypes.byref(pb), igc.F16, A, B, None, None, Cp, float("nan"), 0.0, 0,
                            None) == 1
    assert lib.conv2d_fprop(ctypes.byref(pb), igc.F16, A + 2, B, None, None, Cp, 1.0, 0.0, 0,
                            None) == 3
    assert lib.conv2d_fprop(ctypes.byref(pb), igc.F16, A, B, A + 8, None, Cp, 1.0, 0.0, 0,
                            None) == 3
    assert lib.conv2d_fprop(ctypes.byref(pb), igc.F32, A, B, None, None, Cp, 1.0, 0.0, 0, None) == 2


def test_dgrad_wgrad_int8_reject_invalid(igc):
    lib = igc.load()
    pb = igc.Problem.make(_pb(N=0))
    assert lib.conv2d_dgrad(ctypes.byref(pb), igc.F16, A, B, None, Cp, 1.0, 0.0, None) == 1
    assert lib.conv2d_wgrad(ctypes.byref(pb), igc.F16, igc.F32, A, B, None, Cp, 1.0, 0.0, None, 0,
                            None) == 1
    assert lib.conv2d_fprop_int8(ctypes.byref(pb), A, B, None, Cp, 0.1, 0.1, 0.1, 1, None, 0,
                                 None) == 1
    pb = igc.Problem.make(_pb(stride_h=5, stride_w=4))
    assert lib.conv2d_dgrad(ctypes.byref(pb), igc.F16, A, B, None, Cp, 1.0, 0.0, None) == 2
    pb = igc.Problem.make(_pb())
    assert lib.conv2d_wgrad(ctypes.byref(pb), igc.F16, igc.I8, A, B, None, Cp, 1.0, 0.0, None, 0,
                            None) == 2
    assert lib.conv2d_fprop_int8(ctypes.byref(pb), A, B, None, Cp, 0.0, 0.1, 0.1, 1, None, 0,
                                 None) == 1
    assert lib.conv2d_fprop_int8(ctypes.byref(pb), A, B, None, Cp, 0.1, float("inf"), 0.1, 1, None,
                                 0, None) == 1
    pb = igc.Problem.make(_pb(C=8))   # int8 needs multiples of 16
    assert lib.conv2d_fprop_int8(ctypes.byref(pb), A, B, None, Cp, 0.1, 0.1, 0.1, 1, None, 0,
                                 None) == 2
    pb = igc.Problem.make(_pb(C=512, R=3, S=3))  # R*S*C > 4096: split, int32 partials
    assert lib.conv2d_fprop_int8(ctypes.byref(pb), A, B, None, Cp, 0.1, 0.1, 0.1, 1, None, 0,
                                 None) == 4  # no workspace
    assert igc.conv2d_fprop_int8_workspace_size(_pb(C=512, R=3, S=3)) > \
        2 * 8 * 8 * 512 * 2 + 16 * 9 * 512 * 2
    pb = igc.Problem.make(_pb(C=32))
    assert lib.conv2d_fprop_int8(ctypes.byref(pb), A, B, None, Cp, 0.1, 0.1, 0.1, 1, None, 0,
                                 None) == 4  # no workspace


def test_permutes_reject_invalid(igc):
    lib = igc.load()
    assert lib.nchw_to_nhwc(None, B, 1, 1, 1, 1, 2, None) == 1
    assert lib.nchw_to_nhwc(A, B, 1, 0, 1, 1, 2, None) == 1
    assert lib.nhwc_to_nchw(A, B, 1, 1, 1, 1, 3, None) == 1
    assert lib.nhwc_to_nchw(A + 1, B, 1, 1, 1, 1, 2, None) == 3


def test_workspace_sizes(igc):
    pb = _pb(N=2, H=8, W=8, C=8, K=16)
    ws = igc.conv2d_wgrad_workspace_size(pb, igc.F16, igc.F16)
    assert ws > 0 and ws % 4 == 0
    assert igc.conv2d_wgrad_workspace_size(_pb(N=0), igc.F16, igc.F16) == 0
    assert igc.conv2d_wgrad_workspace_size(pb, igc.F32, igc.F16) == 0
    n = igc.conv2d_fprop_int8_workspace_size(_pb(C=16, K=16))
    assert n >= 2 * (2 * 8 * 8 * 16) + 2 * (16 * 9 * 16)


def test_tuning_keys(igc):
    lib = igc.load()
    assert lib.igconv_set_tuning(igc.TUNE_BLOCK_N, 96) == 1
    assert lib.igconv_set_tuning(99, 1) == 1
    assert lib.igconv_set_tuning(igc.TUNE_WGRAD_SPLITS, -1) == 1
    assert lib.igconv_set_tuning(igc.TUNE_BLOCK_N, 128) == 0
    assert lib.igconv_set_tuning(igc.TUNE_BLOCK_N, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_EPI_GROUPS, 3) == 1
    assert lib.igconv_set_tuning(igc.TUNE_EPI_GROUPS, -1) == 1
    assert lib.igconv_set_tuning(igc.TUNE_EPI_GROUPS, 2) == 0
    assert lib.igconv_set_tuning(igc.TUNE_EPI_GROUPS, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 3) == 1
    assert lib.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 2) == 0
    assert lib.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_CTA_PAIRS, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_FEW_CHANNELS, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_FEW_CHANNELS, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_FEW_CHANNELS, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_RASTER, 65) == 1
    assert lib.igconv_set_tuning(igc.TUNE_RASTER, -1) == 1
    assert lib.igconv_set_tuning(igc.TUNE_RASTER, 8) == 0
    assert lib.igconv_set_tuning(igc.TUNE_RASTER, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_RESIDENT_FILTER, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_RESIDENT_FILTER, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_RESIDENT_FILTER, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_DGRAD_ROWS, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_DGRAD_ROWS, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_DGRAD_ROWS, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_EPILOGUE_KERNEL, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_EPILOGUE_KERNEL, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_EPILOGUE_KERNEL, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_HALO, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_HALO, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_HALO, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_ONE_ISSUER, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_ONE_ISSUER, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_ONE_ISSUER, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_WGRAD_HALO, 0) == 0
    assert lib.igconv_set_tuning(igc.TUNE_PDL, 2) == 1
    assert lib.igconv_set_tuning(igc.TUNE_PDL, -1) == 1
    assert lib.igconv_set_tuning(igc.TUNE_PDL, 1) == 0
    assert lib.igconv_set_tuning(igc.TUNE_PDL, 0) == 0


def test_grouped_reject_invalid(igc):
    lib = igc.load()
    pb = igc.Problem.make(_pb())
    fp = lib.conv2d_grouped_fprop
    # groups < 1, or not dividing C and K: INVALID_ARG
    for g in (0, -1, 3, 32):
        assert fp(ctypes.byref(pb), g, igc.F16, A, B, None, None, Cp, 1.0, 0.0, 0, None) == 1
    # C != K with groups > 1, or a group width outside 1..32: UNSUPPORTED
    pbk = igc.Problem.make(_pb(K=32))
    assert fp(ctypes.byref(pbk), 16, igc.F16, A, B, None, None, Cp, 1.0, 0.0, 0, None) == 2
    pb128 = igc.Problem.make(_pb(C=128, K=128))
    assert fp(ctypes.byref(pb128), 2, igc.F16, A, B, None, None, Cp, 1.0, 0.0, 0, None) == 2
    pb48 = igc.Problem.make(_pb(C=48, K=48))
    assert fp(ctypes.byref(pb48), 2, igc.F16, A, B, None, None, Cp, 1.0, 0.0, 0, None) == 2
    # depthwise: the dense path's validation applies
    pb12 = igc.Problem.make(_pb(C=12, K=12))
    assert fp(ctypes.byref(pb12), 12, igc.F16, A, B, None, None, Cp, 1.0, 0.0, 0, None) == 2
    assert fp(ctypes.byref(pb), 16, igc.F16, None, B, None, None, Cp, 1.0, 0.0, 0, None) == 1
    assert fp(ctypes.byref(pb), 16, igc.F16, A, B, None, None, Cp, 1.0, 1.0, 0, None) == 1
    assert fp(ctypes.byref(pb), 16, igc.F32, A, B, None, None, Cp, 1.0, 0.0, 0, None) == 2
    assert fp(ctypes.byref(pb), 16, igc.F16, A + 4, B, None, None, Cp, 1.0, 0.0, 0, None) == 3
    assert lib.conv2d_grouped_dgrad(ctypes.byref(pb), 3, igc.F16, A, B, None, Cp, 1.0, 0.0,
                                    None) == 1
    assert lib.conv2d_grouped_dgrad(ctypes.byref(pb), 16, igc.F16, A, B, None, Cp + 2, 1.0, 0.0,
                                    None) == 3
    # C != K whose 64-wide tiles would split a group (24 output channels per
    # group): no path at all
    pb_split = igc.Problem.make(_pb(C=24, K=48))
    assert lib.conv2d_grouped_wgrad(ctypes.byref(pb_split), 2, igc.F16, igc.F32, A, B, None, Cp,
                                    1.0, 0.0, None, 0, None) == 2
    assert lib.conv2d_grouped_wgrad(ctypes.byref(pb), 16, igc.F16, igc.I8, A, B, None, Cp, 1.0,
                                    0.0, None, 0, None) == 2
    assert igc.conv2d_grouped_wgrad_workspace_size(_pb(), 5, igc.F16, igc.F32) == 0
    # tensor-core grouped fprop: a workspace (the dense block-diagonal
    # filter, K*R*S*C*2 bytes) for C == K from width 4 and for C != K when
    # the tiles hold whole groups and the windows are multiples of 8
    assert igc.conv2d_grouped_fprop_workspace_size(_pb(C=128, K=128), 32, igc.BF16) >= \
        128 * 9 * 128 * 2
    assert igc.conv2d_grouped_fprop_workspace_size(_pb(C=64, K=128), 16, igc.BF16) >= \
        128 * 9 * 64 * 2
    assert igc.conv2d_grouped_dgrad_workspace_size(_pb(C=128, K=64), 16, igc.BF16) >= \
        64 * 9 * 128 * 2
    assert igc.conv2d_grouped_fprop_workspace_size(_pb(C=24, K=48), 2, igc.BF16) == 0
    # 16 output channels per group of 1 input channel: 4-channel windows
    assert igc.conv2d_grouped_fprop_workspace_size(_pb(C=16, K=256), 16, igc.BF16) == 0
    assert igc.conv2d_grouped_fprop_workspace_size(_pb(C=128, K=128), 64, igc.BF16) == 0
    assert igc.conv2d_grouped_fprop_workspace_size(_pb(C=128, K=128), 2, igc.F32) == 0
    pb128 = igc.Problem.make(_pb(C=128, K=128))
    assert lib.conv2d_grouped_fprop_ws(ctypes.byref(pb128), 32, igc.BF16, A, B, None, None, Cp,
                                       1.0, 0.0, 0, None, 0, None) == 4
    # the binding checks the filter size against C/groups before the call
    with pytest.raises(ValueError):
        igc.conv2d_grouped_fprop(_pb(), 3, igc.F16, None, None, None, None, None)


def test_conv3d_rejects_invalid(igc):
    lib = igc.load()
    base = dict(N=1, D=4, H=8, W=8, C=16, K=16, T=3, R=3, S=3, pad_d=1, pad_h=1, pad_w=1,
                stride_d=1, stride_h=1, stride_w=1, dil_d=1, dil_h=1, dil_w=1)
    def call(**kw):
        pb = igc.Problem3D.make(dict(base, **kw))
        return lib.conv3d_fprop(ctypes.byref(pb), igc.BF16, A, B, None, None, Cp, 1.0, 0.0, 0,
                                None)
    assert call(D=0) == 1
    assert call(pad_d=-1) == 1
    assert call(D=1, T=3, pad_d=0) == 1          # no output depth
    assert call(C=12) == 2
    assert call(pad_d=16) == 2                   # 5D im2col box limit
    assert call(D=20, T=9, dil_d=2) == 2         # dil*(T-1) = 16 > 15
    assert call(stride_d=9) == 2
    assert igc.conv3d_output_size(base) == (4, 8, 8)
    assert igc.conv3d_output_size(dict(base, stride_d=2, pad_d=0)) == (1, 8, 8)
    pb = igc.Problem3D.make(base)
    assert lib.conv3d_fprop(ctypes.byref(pb), igc.BF16, A + 8, B, None, None, Cp, 1.0, 0.0, 0,
                            None) == 3
