"""Python binding of libigconv, the implicit-GEMM convolution library for
GB300 (sm_103a).

Argument marshalling only: every function here forwards to the C entry
point of the same name in ``libigconv.so`` (declared in ``include/igconv.h``);
all arithmetic runs in the library's CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no fallback: if the shared library
has not been built, every call raises ``RuntimeError``.

Tensors are CUDA tensors in NHWC (activations) / KRSC (filters) layout,
contiguous.  Sizes are checked against the problem before the call so that a
mismatched tensor cannot be read or written out of bounds.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "IgconvError", "Problem", "library_path", "load",
    "conv2d_output_size", "conv2d_fprop", "conv2d_fprop_workspace_size", "conv2d_fprop_ws",
    "conv2d_dgrad", "conv2d_dgrad_workspace_size", "conv2d_dgrad_ws", "conv2d_wgrad_workspace_size",
    "conv2d_wgrad", "conv2d_fprop_int8_workspace_size", "conv2d_fprop_int8",
    "conv2d_dgrad_int8_workspace_size", "conv2d_dgrad_int8", "conv2d_wgrad_int8_workspace_size",
    "conv2d_wgrad_int8", "conv2d_fprop_winograd_workspace_size", "conv2d_fprop_winograd",
    "conv2d_grouped_fprop", "conv2d_grouped_fprop_workspace_size", "conv2d_grouped_fprop_ws",
    "conv2d_grouped_dgrad", "conv2d_grouped_dgrad_workspace_size", "conv2d_grouped_dgrad_ws",
    "conv2d_grouped_wgrad_workspace_size",
    "conv2d_grouped_wgrad", "grouped_fprop", "grouped_dgrad", "grouped_wgrad",
    "Problem3D", "conv3d_output_size", "conv3d_fprop", "conv3d_dgrad",
    "conv3d_wgrad_workspace_size", "conv3d_wgrad", "fprop3d", "dgrad3d", "wgrad3d",
    "nchw_to_nhwc", "nhwc_to_nchw", "igconv_get_device_status", "igconv_status_string",
    "igconv_set_tuning", "igconv_selftest_wait_timeout",
    "fprop", "dgrad", "wgrad", "fprop_int8",
    "F16", "BF16", "F32", "I8", "I32",
    "TUNE_WGRAD_SPLITS", "TUNE_BLOCK_N", "TUNE_MAX_CTAS", "TUNE_CTA_PAIRS", "TUNE_EPI_GROUPS",
    "TUNE_CONV_SPLITS", "TUNE_FEW_CHANNELS", "TUNE_RASTER", "TUNE_RESIDENT_FILTER",
    "TUNE_DGRAD_ROWS", "TUNE_EPILOGUE_KERNEL", "TUNE_HALO", "TUNE_ONE_ISSUER", "TUNE_WGRAD_HALO",
    "TUNE_PDL",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libigconv.so")

F16, BF16, F32, I8, I32 = 0, 1, 2, 3, 4
TUNE_WGRAD_SPLITS, TUNE_BLOCK_N, TUNE_MAX_CTAS, TUNE_CTA_PAIRS, TUNE_EPI_GROUPS = 1, 2, 3, 4, 5
TUNE_CONV_SPLITS, TUNE_FEW_CHANNELS, TUNE_RASTER, TUNE_RESIDENT_FILTER = 6, 7, 8, 9
TUNE_DGRAD_ROWS, TUNE_EPILOGUE_KERNEL, TUNE_HALO, TUNE_ONE_ISSUER = 10, 11, 12, 13
TUNE_WGRAD_HALO, TUNE_PDL = 14, 15
STATUS_NAMES = {0: "IGCONV_OK", 1: "IGCONV_ERR_INVALID_ARG", 2: "IGCONV_ERR_UNSUPPORTED",
                3: "IGCONV_ERR_MISALIGNED", 4: "IGCONV_ERR_WORKSPACE", 5: "IGCONV_ERR_CUDA",
                6: "IGCONV_ERR_DEVICE_TIMEOUT"}
_TORCH_CODE = {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32,
               torch.int8: I8, torch.int32: I32}


class IgconvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class Problem(ctypes.Structure):
    """igconv_problem_t."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "N", "H", "W", "C", "K", "R", "S",
        "pad_h", "pad_w", "stride_h", "stride_w", "dil_h", "dil_w")]

    @classmethod
    def make(cls, pb) -> "Problem":
        if isinstance(pb, Problem):
            return pb
        return cls(*[int(pb[n]) for n, _ in cls._fields_])

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class Problem3D(ctypes.Structure):
    """igconv_problem3d_t."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "N", "D", "H", "W", "C", "K", "T", "R", "S", "pad_d", "pad_h", "pad_w",
        "stride_d", "stride_h", "stride_w", "dil_d", "dil_h", "dil_w")]

    @classmethod
    def make(cls, pb) -> "Problem3D":
        if isinstance(pb, Problem3D):
            return pb
        return cls(*[int(pb[n]) for n, _ in cls._fields_])


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libigconv.so (raises RuntimeError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, D, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t
        PP = ctypes.POINTER(Problem)
        sig = {
            "conv2d_output_size": (I, [PP, ctypes.POINTER(I), ctypes.POINTER(I)]),
            "conv2d_fprop": (I, [PP, I, P, P, P, P, P, F, F, I, P]),
            "conv2d_fprop_workspace_size": (SZ, [PP, I]),
            "conv2d_fprop_ws": (I, [PP, I, P, P, P, P, P, F, F, I, P, SZ, P]),
            "conv2d_dgrad": (I, [PP, I, P, P, P, P, F, F, P]),
            "conv2d_dgrad_workspace_size": (SZ, [PP, I]),
            "conv2d_dgrad_ws": (I, [PP, I, P, P, P, P, F, F, P, SZ, P]),
            "conv2d_wgrad_workspace_size": (SZ, [PP, I, I]),
            "conv2d_wgrad": (I, [PP, I, I, P, P, P, P, F, F, P, SZ, P]),
            "conv2d_fprop_int8_workspace_size": (SZ, [PP]),
            "conv2d_fprop_int8": (I, [PP, P, P, P, P, D, D, D, I, P, SZ, P]),
            "conv2d_fprop_winograd_workspace_size": (SZ, [PP, I]),
            "conv2d_fprop_winograd": (I, [PP, I, P, P, P, P, P, F, F, I, P, SZ, P]),
            "conv2d_dgrad_int8_workspace_size": (SZ, [PP]),
            "conv2d_dgrad_int8": (I, [PP, P, P, P, P, SZ, P]),
            "conv2d_wgrad_int8_workspace_size": (SZ, [PP]),
            "conv2d_wgrad_int8": (I, [PP, P, P, P, P, SZ, P]),
            "conv2d_grouped_fprop": (I, [PP, I, I, P, P, P, P, P, F, F, I, P]),
            "conv2d_grouped_fprop_workspace_size": (SZ, [PP, I, I]),
            "conv2d_grouped_fprop_ws": (I, [PP, I, I, P, P, P, P, P, F, F, I, P, SZ, P]),
            "conv2d_grouped_dgrad": (I, [PP, I, I, P, P, P, P, F, F, P]),
            "conv2d_grouped_dgrad_workspace_size": (SZ, [PP, I, I]),
            "conv2d_grouped_dgrad_ws": (I, [PP, I, I, P, P, P, P, F, F, P, SZ, P]),
            "conv2d_grouped_wgrad_workspace_size": (SZ, [PP, I, I, I]),
            "conv2d_grouped_wgrad": (I, [PP, I, I, I, P, P, P, P, F, F, P, SZ, P]),
            "conv3d_output_size": (I, [ctypes.POINTER(Problem3D), ctypes.POINTER(I),
                                       ctypes.POINTER(I), ctypes.POINTER(I)]),
            "conv3d_fprop": (I, [ctypes.POINTER(Problem3D), I, P, P, P, P, P, F, F, I, P]),
            "conv3d_dgrad": (I, [ctypes.POINTER(Problem3D), I, P, P, P, P, F, F, P]),
            "conv3d_wgrad_workspace_size": (SZ, [ctypes.POINTER(Problem3D), I, I]),
            "conv3d_wgrad": (I, [ctypes.POINTER(Problem3D), I, I, P, P, P, P, F, F, P, SZ, P]),
            "nchw_to_nhwc": (I, [P, P, I, I, I, I, I, P]),
            "nhwc_to_nchw": (I, [P, P, I, I, I, I, I, P]),
            "igconv_get_device_status": (I, [P]),
            "igconv_status_string": (ctypes.c_char_p, [I]),
            "igconv_set_tuning": (I, [I, I]),
            "igconv_selftest_wait_timeout": (I, [I, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _check(status: int, where: str) -> None:
    if status != 0:
        raise IgconvError(status, where)


def _dtype_code(dt) -> int:
    if isinstance(dt, int):
        return dt
    return _TORCH_CODE[dt]


def _expect(t, numel: int, name: str) -> None:
    if t is None or isinstance(t, int):
        return
    if t.numel() != numel:
        raise ValueError(f"{name}: expected {numel} elements, got {t.numel()}")


# ---------------------------------------------------------------------------
# The C entry points
# ---------------------------------------------------------------------------

def conv2d_output_size(prob):
    pb = Problem.make(prob)
    P, Q = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().conv2d_output_size(ctypes.byref(pb), ctypes.byref(P), ctypes.byref(Q)),
           "conv2d_output_size")
    return P.value, Q.value


def conv2d_fprop(prob, dtype, X, Wt, bias, Cin, Y, alpha=1.0, beta=0.0, relu=False,
                 stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(Wt, pb.K * pb.R * pb.S * pb.C, "Wt")
    _expect(bias, pb.K, "bias")
    _expect(Y, pb.N * P * Q * pb.K, "Y")
    if beta != 0.0:
        _expect(Cin, pb.N * P * Q * pb.K, "Cin")
    _check(load().conv2d_fprop(ctypes.byref(pb), _dtype_code(dtype), _ptr(X), _ptr(Wt),
                               _ptr(bias), _ptr(Cin) if beta != 0.0 else None, _ptr(Y),
                               float(alpha), float(beta), int(bool(relu)), _stream(stream)),
           "conv2d_fprop")


def conv2d_fprop_workspace_size(prob, dtype) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_fprop_workspace_size(ctypes.byref(pb), _dtype_code(dtype)))


def conv2d_fprop_ws(prob, dtype, X, Wt, bias, Cin, Y, alpha=1.0, beta=0.0, relu=False,
                    workspace=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(Wt, pb.K * pb.R * pb.S * pb.C, "Wt")
    _expect(bias, pb.K, "bias")
    _expect(Y, pb.N * P * Q * pb.K, "Y")
    if beta != 0.0:
        _expect(Cin, pb.N * P * Q * pb.K, "Cin")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_fprop_ws(ctypes.byref(pb), _dtype_code(dtype), _ptr(X), _ptr(Wt),
                                  _ptr(bias), _ptr(Cin) if beta != 0.0 else None, _ptr(Y),
                                  float(alpha), float(beta), int(bool(relu)), _ptr(workspace),
                                  nbytes, _stream(stream)),
           "conv2d_fprop_ws")


def conv2d_dgrad(prob, dtype, dY, Wt, Cin, dX, alpha=1.0, beta=0.0, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(Wt, pb.K * pb.R * pb.S * pb.C, "Wt")
    _expect(dX, pb.N * pb.H * pb.W * pb.C, "dX")
    if beta != 0.0:
        _expect(Cin, pb.N * pb.H * pb.W * pb.C, "Cin")
    _check(load().conv2d_dgrad(ctypes.byref(pb), _dtype_code(dtype), _ptr(dY), _ptr(Wt),
                               _ptr(Cin) if beta != 0.0 else None, _ptr(dX), float(alpha),
                               float(beta), _stream(stream)),
           "conv2d_dgrad")


def conv2d_dgrad_workspace_size(prob, dtype) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_dgrad_workspace_size(ctypes.byref(pb), _dtype_code(dtype)))


def conv2d_dgrad_ws(prob, dtype, dY, Wt, Cin, dX, alpha=1.0, beta=0.0, workspace=None,
                    workspace_bytes=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(Wt, pb.K * pb.R * pb.S * pb.C, "Wt")
    _expect(dX, pb.N * pb.H * pb.W * pb.C, "dX")
    if beta != 0.0:
        _expect(Cin, pb.N * pb.H * pb.W * pb.C, "Cin")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_dgrad_ws(ctypes.byref(pb), _dtype_code(dtype), _ptr(dY), _ptr(Wt),
                                  _ptr(Cin) if beta != 0.0 else None, _ptr(dX), float(alpha),
                                  float(beta), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream)),
           "conv2d_dgrad_ws")


def conv2d_wgrad_workspace_size(prob, dtype, dw_dtype) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_wgrad_workspace_size(ctypes.byref(pb), _dtype_code(dtype),
                                                  _dtype_code(dw_dtype)))


def conv2d_wgrad(prob, dtype, dw_dtype, X, dY, Cin, dW, alpha=1.0, beta=0.0, workspace=None,
                 workspace_bytes=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(dW, pb.K * pb.R * pb.S * pb.C, "dW")
    if beta != 0.0:
        _expect(Cin, pb.K * pb.R * pb.S * pb.C, "Cin")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_wgrad(ctypes.byref(pb), _dtype_code(dtype), _dtype_code(dw_dtype),
                               _ptr(X), _ptr(dY), _ptr(Cin) if beta != 0.0 else None, _ptr(dW),
                               float(alpha), float(beta), _ptr(workspace), int(workspace_bytes),
                               _stream(stream)),
           "conv2d_wgrad")


def conv2d_fprop_int8_workspace_size(prob) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_fprop_int8_workspace_size(ctypes.byref(pb)))


def conv2d_fprop_int8(prob, X, Wt, bias, Y, act_scale, w_scale, out_scale, relu=True,
                      workspace=None, workspace_bytes=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(Wt, pb.K * pb.R * pb.S * pb.C, "Wt")
    _expect(bias, pb.K, "bias")
    _expect(Y, pb.N * P * Q * pb.K, "Y")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_fprop_int8(ctypes.byref(pb), _ptr(X), _ptr(Wt), _ptr(bias), _ptr(Y),
                                    float(act_scale), float(w_scale), float(out_scale),
                                    int(bool(relu)), _ptr(workspace), int(workspace_bytes),
                                    _stream(stream)),
           "conv2d_fprop_int8")


def conv2d_fprop_winograd_workspace_size(prob, dtype) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_fprop_winograd_workspace_size(ctypes.byref(pb), _dtype_code(dtype)))


def conv2d_fprop_winograd(prob, dtype, X, Wt, bias, Cin, Y, alpha=1.0, beta=0.0, relu=False,
                          workspace=None, workspace_bytes=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(Wt, pb.K * pb.R * pb.S * pb.C, "Wt")
    _expect(bias, pb.K, "bias")
    _expect(Y, pb.N * P * Q * pb.K, "Y")
    if beta != 0.0:
        _expect(Cin, pb.N * P * Q * pb.K, "Cin")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_fprop_winograd(ctypes.byref(pb), _dtype_code(dtype), _ptr(X), _ptr(Wt),
                                        _ptr(bias), _ptr(Cin) if beta != 0.0 else None, _ptr(Y),
                                        float(alpha), float(beta), int(bool(relu)),
                                        _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "conv2d_fprop_winograd")


def conv2d_dgrad_int8_workspace_size(prob) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_dgrad_int8_workspace_size(ctypes.byref(pb)))


def conv2d_dgrad_int8(prob, dY, Wt, dX, workspace=None, workspace_bytes=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(Wt, pb.K * pb.R * pb.S * pb.C, "Wt")
    _expect(dX, pb.N * pb.H * pb.W * pb.C, "dX")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_dgrad_int8(ctypes.byref(pb), _ptr(dY), _ptr(Wt), _ptr(dX),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "conv2d_dgrad_int8")


def conv2d_wgrad_int8_workspace_size(prob) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_wgrad_int8_workspace_size(ctypes.byref(pb)))


def conv2d_wgrad_int8(prob, X, dY, dW, workspace=None, workspace_bytes=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(dW, pb.K * pb.R * pb.S * pb.C, "dW")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_wgrad_int8(ctypes.byref(pb), _ptr(X), _ptr(dY), _ptr(dW),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "conv2d_wgrad_int8")


def _group_sizes(pb, groups):
    groups = int(groups)
    if groups < 1 or pb.C % groups or pb.K % groups:
        raise ValueError("groups must divide C and K")
    return pb.C // groups


def conv2d_grouped_fprop(prob, groups, dtype, X, Wt, bias, Cin, Y, alpha=1.0, beta=0.0,
                         relu=False, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    cg = _group_sizes(pb, groups)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(Wt, pb.K * pb.R * pb.S * cg, "Wt")
    _expect(bias, pb.K, "bias")
    _expect(Y, pb.N * P * Q * pb.K, "Y")
    if beta != 0.0:
        _expect(Cin, pb.N * P * Q * pb.K, "Cin")
    _check(load().conv2d_grouped_fprop(ctypes.byref(pb), int(groups), _dtype_code(dtype), _ptr(X),
                                       _ptr(Wt), _ptr(bias), _ptr(Cin) if beta != 0.0 else None,
                                       _ptr(Y), float(alpha), float(beta), int(bool(relu)),
                                       _stream(stream)),
           "conv2d_grouped_fprop")


def conv2d_grouped_fprop_workspace_size(prob, groups, dtype) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_grouped_fprop_workspace_size(ctypes.byref(pb), int(groups),
                                                          _dtype_code(dtype)))


def conv2d_grouped_fprop_ws(prob, groups, dtype, X, Wt, bias, Cin, Y, alpha=1.0, beta=0.0,
                            relu=False, workspace=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    cg = _group_sizes(pb, groups)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(Wt, pb.K * pb.R * pb.S * cg, "Wt")
    _expect(bias, pb.K, "bias")
    _expect(Y, pb.N * P * Q * pb.K, "Y")
    if beta != 0.0:
        _expect(Cin, pb.N * P * Q * pb.K, "Cin")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_grouped_fprop_ws(ctypes.byref(pb), int(groups), _dtype_code(dtype),
                                          _ptr(X), _ptr(Wt), _ptr(bias),
                                          _ptr(Cin) if beta != 0.0 else None, _ptr(Y),
                                          float(alpha), float(beta), int(bool(relu)),
                                          _ptr(workspace), nbytes, _stream(stream)),
           "conv2d_grouped_fprop_ws")


def conv2d_grouped_dgrad(prob, groups, dtype, dY, Wt, Cin, dX, alpha=1.0, beta=0.0,
                         stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    cg = _group_sizes(pb, groups)
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(Wt, pb.K * pb.R * pb.S * cg, "Wt")
    _expect(dX, pb.N * pb.H * pb.W * pb.C, "dX")
    if beta != 0.0:
        _expect(Cin, pb.N * pb.H * pb.W * pb.C, "Cin")
    _check(load().conv2d_grouped_dgrad(ctypes.byref(pb), int(groups), _dtype_code(dtype),
                                       _ptr(dY), _ptr(Wt), _ptr(Cin) if beta != 0.0 else None,
                                       _ptr(dX), float(alpha), float(beta), _stream(stream)),
           "conv2d_grouped_dgrad")


def conv2d_grouped_dgrad_workspace_size(prob, groups, dtype) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_grouped_dgrad_workspace_size(ctypes.byref(pb), int(groups),
                                                          _dtype_code(dtype)))


def conv2d_grouped_dgrad_ws(prob, groups, dtype, dY, Wt, Cin, dX, alpha=1.0, beta=0.0,
                            workspace=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    cg = _group_sizes(pb, groups)
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(Wt, pb.K * pb.R * pb.S * cg, "Wt")
    _expect(dX, pb.N * pb.H * pb.W * pb.C, "dX")
    if beta != 0.0:
        _expect(Cin, pb.N * pb.H * pb.W * pb.C, "Cin")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_grouped_dgrad_ws(ctypes.byref(pb), int(groups), _dtype_code(dtype),
                                          _ptr(dY), _ptr(Wt), _ptr(Cin) if beta != 0.0 else None,
                                          _ptr(dX), float(alpha), float(beta), _ptr(workspace),
                                          nbytes, _stream(stream)),
           "conv2d_grouped_dgrad_ws")


def conv2d_grouped_wgrad_workspace_size(prob, groups, dtype, dw_dtype) -> int:
    pb = Problem.make(prob)
    return int(load().conv2d_grouped_wgrad_workspace_size(ctypes.byref(pb), int(groups),
                                                          _dtype_code(dtype),
                                                          _dtype_code(dw_dtype)))


def conv2d_grouped_wgrad(prob, groups, dtype, dw_dtype, X, dY, Cin, dW, alpha=1.0, beta=0.0,
                         workspace=None, workspace_bytes=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    cg = _group_sizes(pb, groups)
    _expect(X, pb.N * pb.H * pb.W * pb.C, "X")
    _expect(dY, pb.N * P * Q * pb.K, "dY")
    _expect(dW, pb.K * pb.R * pb.S * cg, "dW")
    if beta != 0.0:
        _expect(Cin, pb.K * pb.R * pb.S * cg, "Cin")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv2d_grouped_wgrad(ctypes.byref(pb), int(groups), _dtype_code(dtype),
                                       _dtype_code(dw_dtype), _ptr(X), _ptr(dY),
                                       _ptr(Cin) if beta != 0.0 else None, _ptr(dW),
                                       float(alpha), float(beta), _ptr(workspace),
                                       int(workspace_bytes), _stream(stream)),
           "conv2d_grouped_wgrad")


def conv3d_output_size(prob):
    pb = Problem3D.make(prob)
    D, P, Q = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(load().conv3d_output_size(ctypes.byref(pb), ctypes.byref(D), ctypes.byref(P),
                                     ctypes.byref(Q)), "conv3d_output_size")
    return D.value, P.value, Q.value


def conv3d_fprop(prob, dtype, X, Wt, bias, Cin, Y, alpha=1.0, beta=0.0, relu=False,
                 stream=None):
    pb = Problem3D.make(prob)
    Do, P, Q = conv3d_output_size(pb)
    _expect(X, pb.N * pb.D * pb.H * pb.W * pb.C, "X")
    _expect(Wt, pb.K * pb.T * pb.R * pb.S * pb.C, "Wt")
    _expect(bias, pb.K, "bias")
    _expect(Y, pb.N * Do * P * Q * pb.K, "Y")
    if beta != 0.0:
        _expect(Cin, pb.N * Do * P * Q * pb.K, "Cin")
    _check(load().conv3d_fprop(ctypes.byref(pb), _dtype_code(dtype), _ptr(X), _ptr(Wt),
                               _ptr(bias), _ptr(Cin) if beta != 0.0 else None, _ptr(Y),
                               float(alpha), float(beta), int(bool(relu)), _stream(stream)),
           "conv3d_fprop")


def conv3d_dgrad(prob, dtype, dY, Wt, Cin, dX, alpha=1.0, beta=0.0, stream=None):
    pb = Problem3D.make(prob)
    Do, P, Q = conv3d_output_size(pb)
    _expect(dY, pb.N * Do * P * Q * pb.K, "dY")
    _expect(Wt, pb.K * pb.T * pb.R * pb.S * pb.C, "Wt")
    _expect(dX, pb.N * pb.D * pb.H * pb.W * pb.C, "dX")
    if beta != 0.0:
        _expect(Cin, pb.N * pb.D * pb.H * pb.W * pb.C, "Cin")
    _check(load().conv3d_dgrad(ctypes.byref(pb), _dtype_code(dtype), _ptr(dY), _ptr(Wt),
                               _ptr(Cin) if beta != 0.0 else None, _ptr(dX), float(alpha),
                               float(beta), _stream(stream)),
           "conv3d_dgrad")


def conv3d_wgrad_workspace_size(prob, dtype, dw_dtype) -> int:
    pb = Problem3D.make(prob)
    return int(load().conv3d_wgrad_workspace_size(ctypes.byref(pb), _dtype_code(dtype),
                                                  _dtype_code(dw_dtype)))


def conv3d_wgrad(prob, dtype, dw_dtype, X, dY, Cin, dW, alpha=1.0, beta=0.0, workspace=None,
                 workspace_bytes=None, stream=None):
    pb = Problem3D.make(prob)
    Do, P, Q = conv3d_output_size(pb)
    _expect(X, pb.N * pb.D * pb.H * pb.W * pb.C, "X")
    _expect(dY, pb.N * Do * P * Q * pb.K, "dY")
    _expect(dW, pb.K * pb.T * pb.R * pb.S * pb.C, "dW")
    if beta != 0.0:
        _expect(Cin, pb.K * pb.T * pb.R * pb.S * pb.C, "Cin")
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().conv3d_wgrad(ctypes.byref(pb), _dtype_code(dtype), _dtype_code(dw_dtype),
                               _ptr(X), _ptr(dY), _ptr(Cin) if beta != 0.0 else None, _ptr(dW),
                               float(alpha), float(beta), _ptr(workspace), int(workspace_bytes),
                               _stream(stream)),
           "conv3d_wgrad")


def nchw_to_nhwc(src, dst, N, C, H, W, elem_bytes=None, stream=None):
    if elem_bytes is None:
        elem_bytes = src.element_size()
    _expect(src, N * C * H * W, "src")
    _expect(dst, N * C * H * W, "dst")
    _check(load().nchw_to_nhwc(_ptr(src), _ptr(dst), N, C, H, W, elem_bytes, _stream(stream)),
           "nchw_to_nhwc")


def nhwc_to_nchw(src, dst, N, C, H, W, elem_bytes=None, stream=None):
    if elem_bytes is None:
        elem_bytes = src.element_size()
    _expect(src, N * C * H * W, "src")
    _expect(dst, N * C * H * W, "dst")
    _check(load().nhwc_to_nchw(_ptr(src), _ptr(dst), N, C, H, W, elem_bytes, _stream(stream)),
           "nhwc_to_nchw")


def igconv_get_device_status(stream=None) -> int:
    """Returns the raw status (0 = OK, 6 = a device-side wait ran out)."""
    return int(load().igconv_get_device_status(_stream(stream)))


def igconv_status_string(status: int) -> str:
    return load().igconv_status_string(int(status)).decode()


def igconv_set_tuning(key: int, value: int) -> None:
    _check(load().igconv_set_tuning(int(key), int(value)), "igconv_set_tuning")


def igconv_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    _check(load().igconv_selftest_wait_timeout(int(timeout_us), _stream(stream)),
           "igconv_selftest_wait_timeout")


# ---------------------------------------------------------------------------
# Conveniences: allocate outputs (and workspaces) with torch on the current
# stream, then call the entry point above.
# ---------------------------------------------------------------------------

def fprop(prob, X, Wt, bias=None, Cin=None, alpha=1.0, beta=0.0, relu=False, out=None,
          stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    Y = out if out is not None else torch.empty((pb.N, P, Q, pb.K), dtype=X.dtype, device=X.device)
    if pb.C <= 8:
        # the few-channel path and its workspace (pixel and filter copies)
        ws = torch.empty(max(conv2d_fprop_workspace_size(pb, X.dtype), 16), dtype=torch.uint8,
                         device=X.device)
        conv2d_fprop_ws(pb, X.dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, ws, stream)
    else:
        conv2d_fprop(pb, X.dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, stream)
    return Y


def dgrad(prob, dY, Wt, Cin=None, alpha=1.0, beta=0.0, out=None, stream=None):
    pb = Problem.make(prob)
    dX = out if out is not None else torch.empty((pb.N, pb.H, pb.W, pb.C), dtype=dY.dtype,
                                                 device=dY.device)
    if pb.C < 8:
        # the few-channel path and its workspace (padded filter, fp32 rows)
        ws = torch.empty(max(conv2d_dgrad_workspace_size(pb, dY.dtype), 16), dtype=torch.uint8,
                         device=dY.device)
        conv2d_dgrad_ws(pb, dY.dtype, dY, Wt, Cin, dX, alpha, beta, ws, stream=stream)
    else:
        conv2d_dgrad(pb, dY.dtype, dY, Wt, Cin, dX, alpha, beta, stream)
    return dX


def wgrad(prob, X, dY, dw_dtype=None, Cin=None, alpha=1.0, beta=0.0, out=None, workspace=None,
          stream=None):
    pb = Problem.make(prob)
    dw_dtype = dw_dtype or X.dtype
    dW = out if out is not None else torch.empty((pb.K, pb.R, pb.S, pb.C), dtype=dw_dtype,
                                                 device=X.device)
    if workspace is None:
        need = conv2d_wgrad_workspace_size(pb, X.dtype, dw_dtype)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    conv2d_wgrad(pb, X.dtype, dw_dtype, X, dY, Cin, dW, alpha, beta, workspace, None, stream)
    return dW


def fprop_int8(prob, X, Wt, bias, act_scale, w_scale, out_scale, relu=True, out=None,
               workspace=None, stream=None):
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    Y = out if out is not None else torch.empty((pb.N, P, Q, pb.K), dtype=torch.int8,
                                                device=X.device)
    if workspace is None:
        workspace = torch.empty(max(conv2d_fprop_int8_workspace_size(pb), 16), dtype=torch.uint8,
                                device=X.device)
    conv2d_fprop_int8(pb, X, Wt, bias, Y, act_scale, w_scale, out_scale, relu, workspace, None,
                      stream)
    return Y


def grouped_fprop(prob, groups, X, Wt, bias=None, Cin=None, alpha=1.0, beta=0.0, relu=False,
                  out=None, stream=None):
    """Grouped fprop; allocates the workspace that opens the tensor-core path
    (C == K with group widths from 4, C != K with whole groups per 64-wide
    tile) or the few-channel path (groups = 1, C <= 8)."""
    pb = Problem.make(prob)
    P, Q = conv2d_output_size(pb)
    Y = out if out is not None else torch.empty((pb.N, P, Q, pb.K), dtype=X.dtype, device=X.device)
    need = conv2d_grouped_fprop_workspace_size(pb, groups, X.dtype)
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=X.device)
        conv2d_grouped_fprop_ws(pb, groups, X.dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, ws,
                                stream)
    else:
        conv2d_grouped_fprop(pb, groups, X.dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, stream)
    return Y


def grouped_dgrad(prob, groups, dY, Wt, Cin=None, alpha=1.0, beta=0.0, out=None, stream=None):
    """Grouped dgrad; allocates the workspace that opens the tensor-core path
    (C == K with group widths from 4, C != K with whole groups per 64-wide
    tile)."""
    pb = Problem.make(prob)
    dX = out if out is not None else torch.empty((pb.N, pb.H, pb.W, pb.C), dtype=dY.dtype,
                                                 device=dY.device)
    need = conv2d_grouped_dgrad_workspace_size(pb, groups, dY.dtype)
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=dY.device)
        conv2d_grouped_dgrad_ws(pb, groups, dY.dtype, dY, Wt, Cin, dX, alpha, beta, ws, stream)
    else:
        conv2d_grouped_dgrad(pb, groups, dY.dtype, dY, Wt, Cin, dX, alpha, beta, stream)
    return dX


def grouped_wgrad(prob, groups, X, dY, dw_dtype=None, Cin=None, alpha=1.0, beta=0.0, out=None,
                  workspace=None, stream=None):
    pb = Problem.make(prob)
    dw_dtype = dw_dtype or X.dtype
    cg = _group_sizes(pb, groups)
    dW = out if out is not None else torch.empty((pb.K, pb.R, pb.S, cg), dtype=dw_dtype,
                                                 device=X.device)
    if workspace is None:
        need = conv2d_grouped_wgrad_workspace_size(pb, groups, X.dtype, dw_dtype)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    conv2d_grouped_wgrad(pb, groups, X.dtype, dw_dtype, X, dY, Cin, dW, alpha, beta, workspace,
                         None, stream)
    return dW


def fprop3d(prob, X, Wt, bias=None, Cin=None, alpha=1.0, beta=0.0, relu=False, out=None,
            stream=None):
    pb = Problem3D.make(prob)
    Do, P, Q = conv3d_output_size(pb)
    Y = out if out is not None else torch.empty((pb.N, Do, P, Q, pb.K), dtype=X.dtype,
                                                device=X.device)
    conv3d_fprop(pb, X.dtype, X, Wt, bias, Cin, Y, alpha, beta, relu, stream)
    return Y


def dgrad3d(prob, dY, Wt, Cin=None, alpha=1.0, beta=0.0, out=None, stream=None):
    pb = Problem3D.make(prob)
    dX = out if out is not None else torch.empty((pb.N, pb.D, pb.H, pb.W, pb.C), dtype=dY.dtype,
                                                 device=dY.device)
    conv3d_dgrad(pb, dY.dtype, dY, Wt, Cin, dX, alpha, beta, stream)
    return dX


def wgrad3d(prob, X, dY, dw_dtype=None, Cin=None, alpha=1.0, beta=0.0, out=None, workspace=None,
            stream=None):
    pb = Problem3D.make(prob)
    dw_dtype = dw_dtype or X.dtype
    dW = out if out is not None else torch.empty((pb.K, pb.T, pb.R, pb.S, pb.C), dtype=dw_dtype,
                                                 device=X.device)
    if workspace is None:
        need = conv3d_wgrad_workspace_size(pb, X.dtype, dw_dtype)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    conv3d_wgrad(pb, X.dtype, dw_dtype, X, dY, Cin, dW, alpha, beta, workspace, None, stream)
    return dW
