"""CPU oracle for implicit-GEMM convolution: TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under
``convolution_implicit_gemm_gb300`` never imports it, and the two share no
code.

The arithmetic lives in ``conv_oracle.c`` (plain C, fp64/int64 loops over the
definition of each pass); this module only compiles it with gcc and marshals
numpy arrays through ctypes.

Every function works on float64 (or int8/int64) numpy arrays in NHWC / KRSC
layout.  Sources for each definition are cited in ``conv_oracle.c``.

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):
  out_size        pinned: printed example shapes, hand arithmetic
  fprop           pinned: hand-worked examples, GEMM special case, brute-force
                  im2col+matmul, zero-inserted dilation, subsampled stride,
                  torch CPU float64 conv2d
  dgrad / wgrad   pinned: exact int64 adjoint identities against fprop, torch
                  CPU float64 conv2d_input / conv2d_weight
  grouped_*       pinned: G = 1 against the dense passes, block-diagonal dense
                  filter, per-channel scipy correlate2d (depthwise), hand
                  example with a channel multiplier, exact int64 adjoint
                  identities, torch CPU float64 grouped conv2d
  fprop3d         pinned: depth 1 against the 2D oracle, separable filters
                  against sums of 2D convolutions of depth slices, brute-force
                  im2col + matmul, torch CPU float64 conv3d
  dgrad3d/wgrad3d pinned: exact int64 adjoint identities with fprop3d,
                  depth 1 against the 2D passes, torch float64 autograd
  fprop_int8      pinned: closed-form requantisation cases (ties, saturation,
                  ReLU), exact accumulation against an int64 numpy einsum
  dgrad_int8 /    pinned: equal to the pinned fp64 dgrad / wgrad on the same
  wgrad_int8      integers, exact int64 adjoint identities with fprop_int8's
                  accumulator, hand-computed wrap past 2^31, int64 numpy
                  im2col products
  abs sums (A)    pinned: equal to the passes run on |operands| by im2col /
                  col2im products and torch convolutions (any route but the
                  oracle's loops)
  f16/bf16 round  pinned: numpy float16 conversion, hand-constructed ties
  permutes        pinned: index formula, round trip
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile conv_oracle.c into liboracle.so next to it (gcc, no fast-math,
    no FMA contraction, so the fp64 results are the same on x86 and Arm)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-D_GNU_SOURCE", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "N", "H", "W", "C", "K", "R", "S",
        "pad_h", "pad_w", "stride_h", "stride_w", "dil_h", "dil_w")]


class _Problem3D(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "N", "D", "H", "W", "C", "K", "T", "R", "S", "pad_d", "pad_h", "pad_w",
        "stride_d", "stride_h", "stride_w", "dil_d", "dil_h", "dil_w")]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_D = ctypes.c_double


def _bind(lib):
    lib.oracle_out_size.argtypes = [_I, _I, _I, _I, _I]
    lib.oracle_out_size.restype = _I
    lib.oracle_fprop.argtypes = [ctypes.POINTER(_Problem), _P, _P, _P, _P, _D, _D, _I,
                                 _P, _I64, _P, _P, _I]
    lib.oracle_fprop.restype = _I
    lib.oracle_dgrad.argtypes = [ctypes.POINTER(_Problem), _P, _P, _P, _D, _D,
                                 _P, _I64, _P, _P, _I]
    lib.oracle_dgrad.restype = _I
    lib.oracle_wgrad.argtypes = [ctypes.POINTER(_Problem), _P, _P, _P, _D, _D,
                                 _P, _I64, _P, _P, _I]
    lib.oracle_wgrad.restype = _I
    lib.oracle_grouped.argtypes = [_I, ctypes.POINTER(_Problem), _I, _P, _P, _P, _P, _D, _D, _I,
                                   _P, _I64, _P, _P, _I]
    lib.oracle_grouped.restype = _I
    lib.oracle_fprop3d.argtypes = [ctypes.POINTER(_Problem3D), _P, _P, _P, _P, _D, _D, _I,
                                   _P, _I64, _P, _P, _I]
    lib.oracle_fprop3d.restype = _I
    lib.oracle_backward3d.argtypes = [_I, ctypes.POINTER(_Problem3D), _P, _P, _P, _D, _D, _P,
                                      _I64, _P, _P, _I]
    lib.oracle_backward3d.restype = _I
    lib.oracle_fprop_int8.argtypes = [ctypes.POINTER(_Problem), _P, _P, _P, _D, _D, _D,
                                      _I, _P, _I64, _P, _P, _I]
    lib.oracle_fprop_int8.restype = _I
    lib.oracle_backward_int8.argtypes = [_I, ctypes.POINTER(_Problem), _P, _P, _P, _I64, _P,
                                         _P, _I]
    lib.oracle_backward_int8.restype = _I
    lib.oracle_requant_multiplier.argtypes = [_D, _D, _D]
    lib.oracle_requant_multiplier.restype = ctypes.c_float
    lib.oracle_requant.argtypes = [_I64, ctypes.c_float, _I]
    lib.oracle_requant.restype = _I
    lib.oracle_f64_to_f16_bits.argtypes = [_D]
    lib.oracle_f64_to_f16_bits.restype = ctypes.c_uint16
    lib.oracle_f64_to_bf16_bits.argtypes = [_D]
    lib.oracle_f64_to_bf16_bits.restype = ctypes.c_uint16
    lib.oracle_round_array.argtypes = [_P, _I64, _I, _P]
    lib.oracle_round_array.restype = None
    lib.oracle_nchw_to_nhwc.argtypes = [_P, _P, _I, _I, _I, _I, _I]
    lib.oracle_nchw_to_nhwc.restype = None
    lib.oracle_nhwc_to_nchw.argtypes = [_P, _P, _I, _I, _I, _I, _I]
    lib.oracle_nhwc_to_nchw.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


class use_library:
    """Context manager that points this module at another build of the oracle
    (used by the planted-mistake test, which compiles a mutated copy)."""

    def __init__(self, path: str):
        self._path = path
        self._saved = None

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self._saved = _lib
            _lib = _bind(ctypes.CDLL(self._path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _problem(pb: dict) -> _Problem:
    return _Problem(*[int(pb[n]) for n in (
        "N", "H", "W", "C", "K", "R", "S",
        "pad_h", "pad_w", "stride_h", "stride_w", "dil_h", "dil_w")])


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def out_size(inp: int, pad: int, dil: int, k: int, stride: int) -> int:
    """floor((in + 2*pad - dil*(k-1) - 1)/stride) + 1, or <= 0 if empty."""
    return int(_load().oracle_out_size(inp, pad, dil, k, stride))


def output_hw(pb: dict):
    return (out_size(pb["H"], pb["pad_h"], pb["dil_h"], pb["R"], pb["stride_h"]),
            out_size(pb["W"], pb["pad_w"], pb["dil_w"], pb["S"], pb["stride_w"]))


def _indices(idx, total):
    if idx is None:
        return None, total
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= total):
        raise IndexError("oracle index out of range")
    return idx, idx.size


def fprop(pb: dict, X, Wt, bias=None, Cin=None, alpha=1.0, beta=0.0, relu=False,
          idx=None, nthreads=None, want_abs=False):
    """Y[n,p,q,k] (fp64, unrounded) for the whole output or for linear indices
    ``idx`` into [N,P,Q,K].  With want_abs also returns |alpha|*sum|x*w|."""
    P, Q = output_hw(pb)
    total = pb["N"] * P * Q * pb["K"]
    X, Wt, bias, Cin = _f64(X), _f64(Wt), _f64(bias), _f64(Cin)
    if beta != 0.0 and Cin is None:
        raise ValueError("beta != 0 needs Cin")
    idx, count = _indices(idx, total)
    Y = np.empty(count, np.float64)
    A = np.empty(count, np.float64) if want_abs else None
    rc = _load().oracle_fprop(ctypes.byref(_problem(pb)), _ptr(X), _ptr(Wt), _ptr(bias),
                              _ptr(Cin), alpha, beta, int(bool(relu)), _ptr(idx), count,
                              _ptr(Y), _ptr(A), nthreads or default_threads())
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        Y = Y.reshape(pb["N"], P, Q, pb["K"])
        A = None if A is None else A.reshape(Y.shape)
    return (Y, A) if want_abs else Y


def dgrad(pb: dict, dY, Wt, Cin=None, alpha=1.0, beta=0.0, idx=None, nthreads=None,
          want_abs=False):
    """dX[n,h,w,c] (fp64) for the whole tensor or linear indices into [N,H,W,C]."""
    total = pb["N"] * pb["H"] * pb["W"] * pb["C"]
    dY, Wt, Cin = _f64(dY), _f64(Wt), _f64(Cin)
    if beta != 0.0 and Cin is None:
        raise ValueError("beta != 0 needs Cin")
    idx, count = _indices(idx, total)
    dX = np.empty(count, np.float64)
    A = np.empty(count, np.float64) if want_abs else None
    rc = _load().oracle_dgrad(ctypes.byref(_problem(pb)), _ptr(dY), _ptr(Wt), _ptr(Cin),
                              alpha, beta, _ptr(idx), count, _ptr(dX), _ptr(A),
                              nthreads or default_threads())
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        dX = dX.reshape(pb["N"], pb["H"], pb["W"], pb["C"])
        A = None if A is None else A.reshape(dX.shape)
    return (dX, A) if want_abs else dX


def wgrad(pb: dict, X, dY, Cin=None, alpha=1.0, beta=0.0, idx=None, nthreads=None,
          want_abs=False):
    """dW[k,r,s,c] (fp64) for the whole tensor or linear indices into [K,R,S,C]."""
    total = pb["K"] * pb["R"] * pb["S"] * pb["C"]
    X, dY, Cin = _f64(X), _f64(dY), _f64(Cin)
    if beta != 0.0 and Cin is None:
        raise ValueError("beta != 0 needs Cin")
    idx, count = _indices(idx, total)
    dW = np.empty(count, np.float64)
    A = np.empty(count, np.float64) if want_abs else None
    rc = _load().oracle_wgrad(ctypes.byref(_problem(pb)), _ptr(X), _ptr(dY), _ptr(Cin),
                              alpha, beta, _ptr(idx), count, _ptr(dW), _ptr(A),
                              nthreads or default_threads())
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        dW = dW.reshape(pb["K"], pb["R"], pb["S"], pb["C"])
        A = None if A is None else A.reshape(dW.shape)
    return (dW, A) if want_abs else dW


def _grouped(which, pb, groups, a, b, bias, Cin, alpha, beta, relu, idx, nthreads, want_abs,
             shape):
    a, b, bias, Cin = _f64(a), _f64(b), _f64(bias), _f64(Cin)
    if beta != 0.0 and Cin is None:
        raise ValueError("beta != 0 needs Cin")
    total = int(np.prod(shape))
    idx, count = _indices(idx, total)
    out = np.empty(count, np.float64)
    A = np.empty(count, np.float64) if want_abs else None
    rc = _load().oracle_grouped(which, ctypes.byref(_problem(pb)), int(groups), _ptr(a), _ptr(b),
                                _ptr(bias), _ptr(Cin), alpha, beta, int(bool(relu)), _ptr(idx),
                                count, _ptr(out), _ptr(A), nthreads or default_threads())
    if rc == -2:
        raise ValueError("groups must divide C and K")
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        out = out.reshape(shape)
        A = None if A is None else A.reshape(shape)
    return (out, A) if want_abs else out


def grouped_fprop(pb: dict, groups: int, X, Wt, bias=None, Cin=None, alpha=1.0, beta=0.0,
                  relu=False, idx=None, nthreads=None, want_abs=False):
    """Grouped fprop: Wt is [K][R][S][C/groups]; output channel k reads the
    input channels of group k // (K/groups).  Y [N][P][Q][K] in fp64."""
    P, Q = output_hw(pb)
    return _grouped(0, pb, groups, X, Wt, bias, Cin, alpha, beta, relu, idx, nthreads,
                    want_abs, (pb["N"], P, Q, pb["K"]))


def grouped_dgrad(pb: dict, groups: int, dY, Wt, Cin=None, alpha=1.0, beta=0.0, idx=None,
                  nthreads=None, want_abs=False):
    """Grouped dgrad: dX [N][H][W][C] in fp64 (Wt [K][R][S][C/groups])."""
    return _grouped(1, pb, groups, dY, Wt, None, Cin, alpha, beta, False, idx, nthreads,
                    want_abs, (pb["N"], pb["H"], pb["W"], pb["C"]))


def grouped_wgrad(pb: dict, groups: int, X, dY, Cin=None, alpha=1.0, beta=0.0, idx=None,
                  nthreads=None, want_abs=False):
    """Grouped wgrad: dW [K][R][S][C/groups] in fp64."""
    return _grouped(2, pb, groups, X, dY, None, Cin, alpha, beta, False, idx, nthreads,
                    want_abs, (pb["K"], pb["R"], pb["S"], pb["C"] // groups))


def output_dhw(pb: dict):
    return (out_size(pb["D"], pb["pad_d"], pb["dil_d"], pb["T"], pb["stride_d"]),
            out_size(pb["H"], pb["pad_h"], pb["dil_h"], pb["R"], pb["stride_h"]),
            out_size(pb["W"], pb["pad_w"], pb["dil_w"], pb["S"], pb["stride_w"]))


def fprop3d(pb: dict, X, Wt, bias=None, Cin=None, alpha=1.0, beta=0.0, relu=False, idx=None,
            nthreads=None, want_abs=False):
    """3D fprop: X [N][D][H][W][C], Wt [K][T][R][S][C] -> Y [N][Do][P][Q][K]
    (fp64, unrounded), or the elements at linear indices idx."""
    Do, P, Q = output_dhw(pb)
    total = pb["N"] * Do * P * Q * pb["K"]
    X, Wt, bias, Cin = _f64(X), _f64(Wt), _f64(bias), _f64(Cin)
    if beta != 0.0 and Cin is None:
        raise ValueError("beta != 0 needs Cin")
    idx, count = _indices(idx, total)
    Y = np.empty(count, np.float64)
    A = np.empty(count, np.float64) if want_abs else None
    prob = _Problem3D(*[int(pb[n]) for n, _ in _Problem3D._fields_])
    rc = _load().oracle_fprop3d(ctypes.byref(prob), _ptr(X), _ptr(Wt), _ptr(bias), _ptr(Cin),
                                alpha, beta, int(bool(relu)), _ptr(idx), count, _ptr(Y), _ptr(A),
                                nthreads or default_threads())
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        Y = Y.reshape(pb["N"], Do, P, Q, pb["K"])
        A = None if A is None else A.reshape(Y.shape)
    return (Y, A) if want_abs else Y


def _backward3d(which, pb, a, b, Cin, alpha, beta, idx, nthreads, want_abs, shape):
    a, b, Cin = _f64(a), _f64(b), _f64(Cin)
    if beta != 0.0 and Cin is None:
        raise ValueError("beta != 0 needs Cin")
    idx, count = _indices(idx, int(np.prod(shape)))
    out = np.empty(count, np.float64)
    A = np.empty(count, np.float64) if want_abs else None
    prob = _Problem3D(*[int(pb[n]) for n, _ in _Problem3D._fields_])
    rc = _load().oracle_backward3d(which, ctypes.byref(prob), _ptr(a), _ptr(b), _ptr(Cin), alpha,
                                   beta, _ptr(idx), count, _ptr(out), _ptr(A),
                                   nthreads or default_threads())
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        out = out.reshape(shape)
        A = None if A is None else A.reshape(shape)
    return (out, A) if want_abs else out


def dgrad3d(pb: dict, dY, Wt, Cin=None, alpha=1.0, beta=0.0, idx=None, nthreads=None,
            want_abs=False):
    """3D dgrad: dX [N][D][H][W][C] (fp64)."""
    return _backward3d(1, pb, dY, Wt, Cin, alpha, beta, idx, nthreads, want_abs,
                       (pb["N"], pb["D"], pb["H"], pb["W"], pb["C"]))


def wgrad3d(pb: dict, X, dY, Cin=None, alpha=1.0, beta=0.0, idx=None, nthreads=None,
            want_abs=False):
    """3D wgrad: dW [K][T][R][S][C] (fp64)."""
    return _backward3d(2, pb, X, dY, Cin, alpha, beta, idx, nthreads, want_abs,
                       (pb["K"], pb["T"], pb["R"], pb["S"], pb["C"]))


def fprop_int8(pb: dict, X, Wt, bias, act_scale, w_scale, out_scale, relu=True,
               idx=None, nthreads=None, want_acc=False):
    """int8 Y[n,p,q,k] after exact int64 accumulation, int32 bias (accumulator
    units), optional ReLU and half-even requantisation with saturation."""
    P, Q = output_hw(pb)
    total = pb["N"] * P * Q * pb["K"]
    X = np.ascontiguousarray(X, dtype=np.int8)
    Wt = np.ascontiguousarray(Wt, dtype=np.int8)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.int32)
    idx, count = _indices(idx, total)
    Y = np.empty(count, np.int8)
    acc = np.empty(count, np.int64) if want_acc else None
    rc = _load().oracle_fprop_int8(ctypes.byref(_problem(pb)), _ptr(X), _ptr(Wt), _ptr(bias),
                                   act_scale, w_scale, out_scale, int(bool(relu)), _ptr(idx),
                                   count, _ptr(Y), _ptr(acc), nthreads or default_threads())
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        Y = Y.reshape(pb["N"], P, Q, pb["K"])
        acc = None if acc is None else acc.reshape(Y.shape)
    return (Y, acc) if want_acc else Y


def _backward_int8(which, pb, a, b, idx, nthreads, want_acc, shape):
    a = np.ascontiguousarray(a, dtype=np.int8)
    b = np.ascontiguousarray(b, dtype=np.int8)
    idx, count = _indices(idx, int(np.prod(shape)))
    out = np.empty(count, np.int32)
    acc = np.empty(count, np.int64) if want_acc else None
    rc = _load().oracle_backward_int8(which, ctypes.byref(_problem(pb)), _ptr(a), _ptr(b),
                                      _ptr(idx), count, _ptr(out), _ptr(acc),
                                      nthreads or default_threads())
    if rc != 0:
        raise ValueError("empty output size")
    if idx is None:
        out = out.reshape(shape)
        acc = None if acc is None else acc.reshape(shape)
    return (out, acc) if want_acc else out


def dgrad_int8(pb: dict, dY, Wt, idx=None, nthreads=None, want_acc=False):
    """int8 dgrad: dX [N][H][W][C] int32 (the exact sum modulo 2^32); with
    want_acc also the exact int64 sums."""
    return _backward_int8(1, pb, dY, Wt, idx, nthreads, want_acc,
                          (pb["N"], pb["H"], pb["W"], pb["C"]))


def wgrad_int8(pb: dict, X, dY, idx=None, nthreads=None, want_acc=False):
    """int8 wgrad: dW [K][R][S][C] int32 (the exact sum modulo 2^32); with
    want_acc also the exact int64 sums."""
    return _backward_int8(2, pb, X, dY, idx, nthreads, want_acc,
                          (pb["K"], pb["R"], pb["S"], pb["C"]))


def requant_multiplier(act_scale: float, w_scale: float, out_scale: float) -> float:
    return float(_load().oracle_requant_multiplier(act_scale, w_scale, out_scale))


def requant(t: int, M: float, relu: bool) -> int:
    return int(_load().oracle_requant(int(t), M, int(bool(relu))))


def f64_to_f16_bits(v: float) -> int:
    return int(_load().oracle_f64_to_f16_bits(float(v)))


def f64_to_bf16_bits(v: float) -> int:
    return int(_load().oracle_f64_to_bf16_bits(float(v)))


def round_bits(v, dtype: str) -> np.ndarray:
    """Round fp64 values to fp16 ('f16') or bf16 ('bf16') bit patterns (uint16),
    nearest-even."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_round_array(_ptr(v), v.size, 1 if dtype == "bf16" else 0, _ptr(out))
    return out


def bits_to_f64(bits, dtype: str) -> np.ndarray:
    """Decode fp16/bf16 bit patterns to float64 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    f32 = (bits.astype(np.uint32) << 16).view(np.float32)
    return f32.astype(np.float64)


def nchw_to_nhwc(src: np.ndarray) -> np.ndarray:
    N, C, H, W = src.shape
    src = np.ascontiguousarray(src)
    dst = np.empty((N, H, W, C), src.dtype)
    _load().oracle_nchw_to_nhwc(_ptr(src), _ptr(dst), N, C, H, W, src.itemsize)
    return dst


def nhwc_to_nchw(src: np.ndarray) -> np.ndarray:
    N, H, W, C = src.shape
    src = np.ascontiguousarray(src)
    dst = np.empty((N, C, H, W), src.dtype)
    _load().oracle_nhwc_to_nchw(_ptr(src), _ptr(dst), N, C, H, W, src.itemsize)
    return dst
