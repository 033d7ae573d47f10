"""ctypes wrapper around the fp64 C oracle (ct_oracle.c).

TEST INFRASTRUCTURE ONLY.  The product (the CUDA library and its binding)
never imports this module.  It shares no code with the CUDA path; the only
thing both sides share is the seeded input generator, which holds none of the
method's arithmetic.

The oracle is the scatter-add of "feat(ops): implement convTranspose2d -- CPU
kernel, backward and StableHLO lowering" (SKaiNET #1464, Summary,
DefaultCpuOps), generalised to 1-D/3-D, groups, asymmetric padding and
output_padding as the ONNX and NKI pages describe.  Inputs are widened to
float64 exactly (bf16/fp16/fp32 values are all representable in double).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ct_oracle.c")
_LIB = os.path.join(_HERE, "libct_oracle.so")
_lib_handle = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ct_oracle.c into libct_oracle.so beside it (plain gcc, -O2).

    No fast-math and no FMA contraction, so the oracle gives the same bits on
    x86 and Arm hosts.
    """
    stale = (not os.path.exists(_LIB)) or (
        os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
            "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        lib.oracle_out_shape.restype = ctypes.c_int
        lib.oracle_out_shape.argtypes = [ctypes.c_int] + [_i64p] * 8
        lib.oracle_conv_transpose_f64.restype = ctypes.c_int
        lib.oracle_conv_transpose_f64.argtypes = (
            [_f64p] * 4 + [ctypes.c_int] + [ctypes.c_int64] * 4 + [_i64p] * 7
            + [ctypes.c_int])
        lib.oracle_conv_transpose_backward_f64.restype = ctypes.c_int
        lib.oracle_conv_transpose_backward_f64.argtypes = (
            [_f64p] * 6 + [ctypes.c_int] + [ctypes.c_int64] * 4 + [_i64p] * 7
            + [ctypes.c_int])
        lib.oracle_activation_f64.restype = ctypes.c_int
        lib.oracle_activation_f64.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int, ctypes.c_double]
        lib.oracle_points_f64.restype = ctypes.c_int
        lib.oracle_points_f64.argtypes = (
            [_f64p] * 3 + [ctypes.c_int] + [ctypes.c_int64] * 4 + [_i64p] * 7
            + [_i64p, ctypes.c_int64, _f64p])
        _lib_handle = lib
    return _lib_handle


def _arr64(vals, nd, name):
    vals = [int(v) for v in vals]
    if len(vals) != nd:
        raise ValueError(f"{name} needs {nd} values, got {len(vals)}")
    a = np.ascontiguousarray(np.array(vals, dtype=np.int64))
    return a


def _ip(a):
    return a.ctypes.data_as(_i64p)


def _fp(a):
    return None if a is None else a.ctypes.data_as(_f64p)


def to_f64(t) -> np.ndarray:
    """Widen a torch tensor or numpy array to a contiguous float64 ndarray.

    Widening from bf16/fp16/fp32 is exact, so the oracle sees exactly the
    values the device sees.
    """
    if t is None:
        return None
    if hasattr(t, "detach"):  # torch tensor
        import torch
        t = t.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _norm(nd, stride, pad_lo, pad_hi, dilation, output_padding):
    one = [1] * nd
    zero = [0] * nd
    return (_arr64(stride if stride is not None else one, nd, "stride"),
            _arr64(pad_lo if pad_lo is not None else zero, nd, "pad_lo"),
            _arr64(pad_hi if pad_hi is not None else zero, nd, "pad_hi"),
            _arr64(dilation if dilation is not None else one, nd, "dilation"),
            _arr64(output_padding if output_padding is not None else zero, nd,
                   "output_padding"))


def out_shape(in_spatial, k, stride=None, pad_lo=None, pad_hi=None,
              dilation=None, output_padding=None):
    """Output spatial extents, (I-1)*s - pad_lo - pad_hi + d*(k-1) + op + 1.

    Raises ValueError when an extent would be < 1 or an argument is invalid.
    """
    nd = len(in_spatial)
    I = _arr64(in_spatial, nd, "in_spatial")
    K = _arr64(k, nd, "k")
    S, PL, PH, DL, OP = _norm(nd, stride, pad_lo, pad_hi, dilation,
                              output_padding)
    out = np.zeros(nd, dtype=np.int64)
    rc = _lib().oracle_out_shape(nd, _ip(I), _ip(K), _ip(S), _ip(PL), _ip(PH),
                                 _ip(DL), _ip(OP), _ip(out))
    if rc != 0:
        raise ValueError(f"oracle_out_shape rejected the arguments (code {rc})")
    return tuple(int(v) for v in out)


def conv_transpose(x, w, bias=None, stride=None, pad_lo=None, pad_hi=None,
                   dilation=None, output_padding=None, groups=1, threads=None):
    """y = ConvTranspose(x, w, bias) in float64 (full scatter-add).

    x: [B, C_in, *spatial], w: [C_in, C_out/groups, *k], bias: [C_out] or None.
    Returns a float64 ndarray [B, C_out, *out_spatial].
    """
    xd, wd, bd = to_f64(x), to_f64(w), to_f64(bias)
    nd = xd.ndim - 2
    if nd < 1 or nd > 3 or wd.ndim != nd + 2:
        raise ValueError("x must be [B, C_in, *spatial] with 1-3 spatial axes "
                         "and w [C_in, C_out/groups, *k]")
    B, C_in = xd.shape[0], xd.shape[1]
    C_out = wd.shape[1] * groups
    if wd.shape[0] != C_in:
        raise ValueError("w.shape[0] must equal C_in")
    if bd is not None and bd.shape != (C_out,):
        raise ValueError("bias must be [C_out]")
    I = _arr64(xd.shape[2:], nd, "in_spatial")
    K = _arr64(wd.shape[2:], nd, "k")
    S, PL, PH, DL, OP = _norm(nd, stride, pad_lo, pad_hi, dilation,
                              output_padding)
    O = out_shape(I, K, S, PL, PH, DL, OP)
    y = np.empty((B, C_out) + O, dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = _lib().oracle_conv_transpose_f64(
        _fp(xd), _fp(wd), _fp(bd), _fp(y), nd, B, C_in, C_out, groups,
        _ip(I), _ip(K), _ip(S), _ip(PL), _ip(PH), _ip(DL), _ip(OP),
        int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return y


def points(x, w, bias, idx, stride=None, pad_lo=None, pad_hi=None,
           dilation=None, output_padding=None, groups=1):
    """y at selected output coordinates, evaluated one by one in float64.

    idx: integer array [n, 2 + nd] of (b, oc, o_1, ..., o_nd).
    """
    xd, wd, bd = to_f64(x), to_f64(w), to_f64(bias)
    nd = xd.ndim - 2
    B, C_in = xd.shape[0], xd.shape[1]
    C_out = wd.shape[1] * groups
    I = _arr64(xd.shape[2:], nd, "in_spatial")
    K = _arr64(wd.shape[2:], nd, "k")
    S, PL, PH, DL, OP = _norm(nd, stride, pad_lo, pad_hi, dilation,
                              output_padding)
    idx = np.asarray(idx, dtype=np.int64).reshape(-1, 2 + nd)
    n = idx.shape[0]
    full = np.zeros((n, 5), dtype=np.int64)
    full[:, 0:2] = idx[:, 0:2]
    full[:, 5 - nd:] = idx[:, 2:]
    full = np.ascontiguousarray(full)
    out = np.empty(n, dtype=np.float64)
    rc = _lib().oracle_points_f64(
        _fp(xd), _fp(wd), _fp(bd), nd, B, C_in, C_out, groups, _ip(I), _ip(K),
        _ip(S), _ip(PL), _ip(PH), _ip(DL), _ip(OP), _ip(full), n, _fp(out))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def conv_transpose_backward(x, w, dy, stride=None, pad_lo=None, pad_hi=None,
                            dilation=None, output_padding=None, groups=1,
                            threads=None, need=("dx", "dw", "db")):
    """(dx, dw, db) for y = ConvTranspose(x, w, bias) and upstream gradient dy,
    in float64: the adjoint of the scatter-add (SKaiNET #1464, Summary,
    convTranspose2dBackward: input, weight and bias gradients).  Entries not
    in `need` are None.
    """
    xd, wd, dyd = to_f64(x), to_f64(w), to_f64(dy)
    nd = xd.ndim - 2
    if nd < 1 or nd > 3 or wd.ndim != nd + 2 or dyd.ndim != nd + 2:
        raise ValueError("x, dy must be [B, C, *spatial] and w [C_in, C_out/groups, *k]")
    B, C_in = xd.shape[0], xd.shape[1]
    C_out = wd.shape[1] * groups
    I = _arr64(xd.shape[2:], nd, "in_spatial")
    K = _arr64(wd.shape[2:], nd, "k")
    S, PL, PH, DL, OP = _norm(nd, stride, pad_lo, pad_hi, dilation, output_padding)
    O = out_shape(I, K, S, PL, PH, DL, OP)
    if dyd.shape != (B, C_out) + O:
        raise ValueError(f"dy must have the output shape {(B, C_out) + O}")
    dx = np.empty(xd.shape, dtype=np.float64) if "dx" in need else None
    dw = np.empty(wd.shape, dtype=np.float64) if "dw" in need else None
    db = np.empty((C_out,), dtype=np.float64) if "db" in need else None
    if threads is None:
        threads = os.cpu_count() or 1
    rc = _lib().oracle_conv_transpose_backward_f64(
        _fp(xd), _fp(wd), _fp(dyd), _fp(dx), _fp(dw), _fp(db), nd, B, C_in, C_out,
        groups, _ip(I), _ip(K), _ip(S), _ip(PL), _ip(PH), _ip(DL), _ip(OP), int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return dx, dw, db


ACTIVATIONS = {"none": 0, "relu": 1, "leaky_relu": 2, "silu": 3, "gelu": 4, "tanh": 5,
               "sigmoid": 6}


def activation(y, act, alpha=0.01):
    """act(y) in float64 (a new array), as oracle_activation_f64 defines it:
    the activation the NKI page applies after the convolution."""
    code = ACTIVATIONS[act] if isinstance(act, str) else int(act)
    out = np.ascontiguousarray(np.array(y, dtype=np.float64, copy=True))
    rc = _lib().oracle_activation_f64(_fp(out), out.size, code, float(alpha))
    if rc != 0:
        raise ValueError(f"unknown activation {act!r}")
    return out
