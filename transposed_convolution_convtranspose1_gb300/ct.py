"""ctypes binding of libct.so (include/ct.h), names as in the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  If
libct.so has not been built, every entry point raises RuntimeError; there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libct.so")

CT_F32, CT_F16, CT_BF16 = 0, 1, 2
CT_OK = 0
CT_ERR_NULL, CT_ERR_RANK, CT_ERR_SHAPE, CT_ERR_PARAM, CT_ERR_GROUPS = 1, 2, 3, 4, 5
CT_ERR_BIAS, CT_ERR_DTYPE, CT_ERR_CUDA, CT_ERR_DEVICE_TIMEOUT = 6, 7, 8, 9
CT_ERR_WORKSPACE, CT_ERR_ALIGN, CT_ERR_ROUTE, CT_ERR_TOO_LARGE = 10, 11, 12, 13

CT_ROUTE_AUTO = -1
CT_ROUTE_NONE = 0
CT_ROUTE_BIAS_FILL = 1
CT_ROUTE_GATHER = 2
CT_ROUTE_GROUPED = 3
CT_ROUTE_SIMT_GEMM = 4
CT_ROUTE_TC_GEMM = 5
CT_ROUTE_TC32_GEMM = 6
ROUTE_NAMES = {0: "none", 1: "bias_fill", 2: "gather", 3: "grouped",
               4: "simt_gemm", 5: "tc_gemm", 6: "tc32_gemm"}

_DTYPE_CODE = {torch.float32: CT_F32, torch.float16: CT_F16, torch.bfloat16: CT_BF16}
# Any other torch dtype is passed as an out-of-range code, which the library
# rejects with CT_ERR_DTYPE.
_BAD_DTYPE_CODE = 99

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int)
_vp = ctypes.c_void_p

EXPORTS = ("ct_version", "ct_last_error", "ct_status_string",
           "ct_conv_transpose_out_shape", "ct_conv_transpose_workspace_bytes",
           "ct_conv_transpose_route", "ct_conv_transpose_route_workspace_bytes",
           "ct_conv_transpose_kernel",
           "ct_conv_transpose_nd", "ct_conv_transpose_nd_route",
           "ct_conv_transpose_nd_host", "ct_conv_transpose_nd_profiled",
           "ct_conv_transpose_nd_noalloc", "ct_device_status", "ct_host_buffers_release",
           "ct_conv_transpose_backward_nd", "ct_conv_transpose_backward_workspace_bytes",
           "ct_conv_transpose_backward_kernels",
           "ct_conv_transpose_nd_ex", "ct_conv_transpose_ex_workspace_bytes",
           "ct_set_wait_limit_ns")

# Size of the static scratch behind ct_conv_transpose_nd_noalloc (CT_NOALLOC_SCRATCH_BYTES).
CT_NOALLOC_SCRATCH_BYTES = 64 << 20


# ct_activation and ct_weight_layout (include/ct.h)
CT_ACT_NONE, CT_ACT_RELU, CT_ACT_LEAKY_RELU, CT_ACT_SILU = 0, 1, 2, 3
CT_ACT_GELU, CT_ACT_TANH, CT_ACT_SIGMOID = 4, 5, 6
ACTIVATIONS = {"none": 0, "relu": 1, "leaky_relu": 2, "silu": 3, "gelu": 4, "tanh": 5,
               "sigmoid": 6}
CT_W_TORCH, CT_W_KDHW_CI_CO, CT_W_KDHW_CO_CI = 0, 1, 2


class CtError(RuntimeError):
    """A nonzero ct_status from the library."""

    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_TEXT.get(status, status)}: {msg}")
        self.status = status


_STATUS_TEXT = {0: "CT_OK", 1: "CT_ERR_NULL", 2: "CT_ERR_RANK", 3: "CT_ERR_SHAPE",
                4: "CT_ERR_PARAM", 5: "CT_ERR_GROUPS", 6: "CT_ERR_BIAS", 7: "CT_ERR_DTYPE",
                8: "CT_ERR_CUDA", 9: "CT_ERR_DEVICE_TIMEOUT", 10: "CT_ERR_WORKSPACE",
                11: "CT_ERR_ALIGN", 12: "CT_ERR_ROUTE", 13: "CT_ERR_TOO_LARGE"}

_lock = threading.Lock()
_lib_handle = None

_AXIS_ARGS = [_i64p, _i64p, _i32p, _i32p, _i32p, _i32p, _i32p]
_SHAPE_ARGS = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + _AXIS_ARGS + [
    ctypes.c_int, ctypes.c_int]


def _declare(h):
    h.ct_version.restype = ctypes.c_int
    h.ct_version.argtypes = []
    h.ct_last_error.restype = ctypes.c_char_p
    h.ct_last_error.argtypes = []
    h.ct_status_string.restype = ctypes.c_char_p
    h.ct_status_string.argtypes = [ctypes.c_int]
    h.ct_conv_transpose_out_shape.restype = ctypes.c_int
    h.ct_conv_transpose_out_shape.argtypes = [ctypes.c_int] + _AXIS_ARGS + [_i64p]
    h.ct_conv_transpose_workspace_bytes.restype = ctypes.c_int
    h.ct_conv_transpose_workspace_bytes.argtypes = _SHAPE_ARGS + [ctypes.POINTER(ctypes.c_size_t)]
    h.ct_conv_transpose_route_workspace_bytes.restype = ctypes.c_int
    h.ct_conv_transpose_route_workspace_bytes.argtypes = _SHAPE_ARGS + [
        ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    h.ct_conv_transpose_route.restype = ctypes.c_int
    h.ct_conv_transpose_route.argtypes = _SHAPE_ARGS + [_i32p]
    h.ct_conv_transpose_kernel.restype = ctypes.c_int
    h.ct_conv_transpose_kernel.argtypes = _SHAPE_ARGS + [ctypes.POINTER(ctypes.c_char_p)]
    h.ct_conv_transpose_backward_kernels.restype = ctypes.c_int
    h.ct_conv_transpose_backward_kernels.argtypes = _SHAPE_ARGS + [ctypes.POINTER(ctypes.c_char_p)] * 2
    h.ct_conv_transpose_nd.restype = ctypes.c_int
    h.ct_conv_transpose_nd.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t] + _SHAPE_ARGS + [_vp]
    h.ct_conv_transpose_nd_route.restype = ctypes.c_int
    h.ct_conv_transpose_nd_route.argtypes = ([_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t]
                                             + _SHAPE_ARGS + [ctypes.c_int, _vp])
    h.ct_conv_transpose_nd_profiled.restype = ctypes.c_int
    h.ct_conv_transpose_nd_profiled.argtypes = ([_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t]
                                                + _SHAPE_ARGS + [ctypes.c_int, _vp, _vp, _vp,
                                                                 _i32p, _i32p])
    h.ct_conv_transpose_nd_host.restype = ctypes.c_int
    h.ct_conv_transpose_nd_host.argtypes = [_vp, _vp, _vp, _vp] + _SHAPE_ARGS + [_vp]
    h.ct_conv_transpose_nd_noalloc.restype = ctypes.c_int
    h.ct_conv_transpose_nd_noalloc.argtypes = [_vp, _vp, _vp, _vp] + _SHAPE_ARGS + [_vp]
    h.ct_set_wait_limit_ns.restype = ctypes.c_ulonglong
    h.ct_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    h.ct_device_status.restype = ctypes.c_int
    h.ct_device_status.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint)]
    h.ct_host_buffers_release.restype = ctypes.c_int
    h.ct_host_buffers_release.argtypes = []
    h.ct_conv_transpose_nd_ex.restype = ctypes.c_int
    h.ct_conv_transpose_nd_ex.argtypes = ([_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t] + _SHAPE_ARGS
                                          + [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_float, _vp])
    h.ct_conv_transpose_ex_workspace_bytes.restype = ctypes.c_int
    h.ct_conv_transpose_ex_workspace_bytes.argtypes = _SHAPE_ARGS + [
        ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    h.ct_conv_transpose_backward_nd.restype = ctypes.c_int
    h.ct_conv_transpose_backward_nd.argtypes = ([_vp] * 7 + [ctypes.c_size_t] + _SHAPE_ARGS + [_vp])
    h.ct_conv_transpose_backward_workspace_bytes.restype = ctypes.c_int
    h.ct_conv_transpose_backward_workspace_bytes.argtypes = _SHAPE_ARGS + [
        ctypes.POINTER(ctypes.c_size_t)]


def lib():
    """The loaded libct.so (loaded on first use; raises if it is missing)."""
    global _lib_handle
    if _lib_handle is None:
        with _lock:
            if _lib_handle is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is not built; run __graft_entry__.build() "
                        "(nvcc for sm_103a). There is no CPU fallback.")
                h = ctypes.CDLL(LIB_PATH)
                _declare(h)
                _lib_handle = h
    return _lib_handle


def _check(rc: int):
    if rc != CT_OK:
        raise CtError(rc, lib().ct_last_error().decode())


def ct_version() -> int:
    return lib().ct_version()


def ct_last_error() -> str:
    return lib().ct_last_error().decode()


def ct_status_string(status: int) -> str:
    return lib().ct_status_string(int(status)).decode()


class _Axes:
    """Per-axis attribute arrays in the ABI's types (kept alive for the call)."""

    def __init__(self, nd, in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding):
        def vec(v, default, ctype):
            if v is None:
                v = default
            if isinstance(v, int):
                v = [v] * nd
            v = [int(a) for a in v]
            if len(v) != nd:
                raise ValueError(f"expected {nd} per-axis values, got {v}")
            return (ctype * max(nd, 1))(*v)

        self.nd = nd
        self.I = vec(in_spatial, 0, ctypes.c_int64)
        self.K = vec(k, 1, ctypes.c_int64)
        self.S = vec(stride, 1, ctypes.c_int)
        self.PL = vec(pad_lo, 0, ctypes.c_int)
        self.PH = vec(pad_hi, 0, ctypes.c_int)
        self.D = vec(dilation, 1, ctypes.c_int)
        self.OP = vec(output_padding, 0, ctypes.c_int)

    def args(self):
        c = ctypes.cast
        return [c(self.I, _i64p), c(self.K, _i64p), c(self.S, _i32p), c(self.PL, _i32p),
                c(self.PH, _i32p), c(self.D, _i32p), c(self.OP, _i32p)]


def dtype_code(dt: torch.dtype) -> int:
    return _DTYPE_CODE.get(dt, _BAD_DTYPE_CODE)


def _shape_args(B, C_in, C_out, ax, groups, dtype):
    return [ax.nd, int(B), int(C_in), int(C_out), *ax.args(), int(groups), int(dtype)]


def ct_conv_transpose_out_shape(in_spatial: Sequence[int], k: Sequence[int], stride=None,
                                pad_lo=None, pad_hi=None, dilation=None, output_padding=None):
    nd = len(in_spatial)
    ax = _Axes(nd, in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding)
    out = (ctypes.c_int64 * max(nd, 1))()
    _check(lib().ct_conv_transpose_out_shape(nd, *ax.args(), ctypes.cast(out, _i64p)))
    return tuple(int(out[i]) for i in range(nd))


def ct_conv_transpose_workspace_bytes(B, C_in, C_out, in_spatial, k, stride=None, pad_lo=None,
                                      pad_hi=None, dilation=None, output_padding=None, groups=1,
                                      dtype=CT_F32, route=CT_ROUTE_AUTO) -> int:
    ax = _Axes(len(in_spatial), in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding)
    n = ctypes.c_size_t(0)
    if route == CT_ROUTE_AUTO:
        rc = lib().ct_conv_transpose_workspace_bytes(
            *_shape_args(B, C_in, C_out, ax, groups, dtype), ctypes.byref(n))
    else:
        rc = lib().ct_conv_transpose_route_workspace_bytes(
            *_shape_args(B, C_in, C_out, ax, groups, dtype), int(route), ctypes.byref(n))
    _check(rc)
    return int(n.value)


def ct_conv_transpose_route(B, C_in, C_out, in_spatial, k, stride=None, pad_lo=None, pad_hi=None,
                            dilation=None, output_padding=None, groups=1, dtype=CT_F32) -> int:
    ax = _Axes(len(in_spatial), in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding)
    r = ctypes.c_int(-1)
    _check(lib().ct_conv_transpose_route(*_shape_args(B, C_in, C_out, ax, groups, dtype),
                                         ctypes.byref(r)))
    return int(r.value)


def ct_conv_transpose_kernel(B, C_in, C_out, in_spatial, k, stride=None, pad_lo=None, pad_hi=None,
                             dilation=None, output_padding=None, groups=1, dtype=CT_F32) -> str:
    """Name of the kernel that dominates ct_conv_transpose_nd's device time here."""
    ax = _Axes(len(in_spatial), in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding)
    name = ctypes.c_char_p()
    _check(lib().ct_conv_transpose_kernel(*_shape_args(B, C_in, C_out, ax, groups, dtype),
                                          ctypes.byref(name)))
    return name.value.decode() if name.value is not None else ""


def ct_conv_transpose_backward_kernels(B, C_in, C_out, in_spatial, k, stride=None, pad_lo=None,
                                       pad_hi=None, dilation=None, output_padding=None, groups=1,
                                       dtype=CT_F32):
    """Names of the kernels that dominate the input and weight gradients' device time: (dx, dw)."""
    ax = _Axes(len(in_spatial), in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding)
    dx, dw = ctypes.c_char_p(), ctypes.c_char_p()
    _check(lib().ct_conv_transpose_backward_kernels(*_shape_args(B, C_in, C_out, ax, groups, dtype),
                                                    ctypes.byref(dx), ctypes.byref(dw)))
    return tuple(n.value.decode() if n.value is not None else "" for n in (dx, dw))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the C ABI must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def _problem_from_tensors(x, w, groups):
    nd = x.dim() - 2
    if nd < 1 or w.dim() != x.dim():
        raise CtError(CT_ERR_RANK, "x must be [B, C_in, *spatial] and w [C_in, C_out/groups, *k]")
    return nd, x.shape[0], x.shape[1], w.shape[1] * groups, tuple(x.shape[2:]), tuple(w.shape[2:])


def _same_device(*tensors) -> torch.device:
    """The one CUDA device all given tensors (None skipped) live on."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise CtError(CT_ERR_PARAM, f"tensors must share one device, got {sorted(map(str, devs))}")
    d = devs.pop()
    if d.type != "cuda":
        raise CtError(CT_ERR_PARAM, f"device tensors expected, got {d}")
    return d


def _stream_handle(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return stream


def ct_conv_transpose_nd(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                         y: torch.Tensor, workspace: Optional[torch.Tensor] = None, stride=None,
                         pad_lo=None, pad_hi=None, dilation=None, output_padding=None,
                         groups: int = 1, route: int = CT_ROUTE_AUTO, stream=None) -> None:
    """Run the device entry point on torch CUDA tensors (y is overwritten).

    route = CT_ROUTE_AUTO calls ct_conv_transpose_nd; any other value calls
    ct_conv_transpose_nd_route with that route.
    """
    nd, B, C_in, C_out, I, K = _problem_from_tensors(x, w, groups)
    if bias is not None and tuple(bias.shape) != (C_out,):
        raise CtError(CT_ERR_BIAS, f"bias must have shape [{C_out}], got {tuple(bias.shape)}")
    for t in (w, bias, y):
        if t is not None and t.dtype != x.dtype:
            raise CtError(CT_ERR_DTYPE, "x, w, bias and y must share one dtype")
    ax = _Axes(nd, I, K, stride, pad_lo, pad_hi, dilation, output_padding)
    if dtype_code(x.dtype) == _BAD_DTYPE_CODE:
        # an unsupported element type: the library's validation names it
        r = ctypes.c_int(-1)
        _check(lib().ct_conv_transpose_route(*_shape_args(B, C_in, C_out, ax, groups,
                                                          _BAD_DTYPE_CODE), ctypes.byref(r)))
    dev = _same_device(x, w, bias, y, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = [_ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(workspace), ws_bytes,
            *_shape_args(B, C_in, C_out, ax, groups, dtype_code(x.dtype))]
    with torch.cuda.device(dev):  # the library works on the current device
        s = _stream_handle(stream, dev)
        if route == CT_ROUTE_AUTO:
            rc = lib().ct_conv_transpose_nd(*args, s)
        else:
            rc = lib().ct_conv_transpose_nd_route(*args, int(route), s)
    _check(rc)


def ct_conv_transpose_nd_profiled(x, w, bias, y, workspace=None, stride=None, pad_lo=None,
                                  pad_hi=None, dilation=None, output_padding=None, groups=1,
                                  route=CT_ROUTE_AUTO, stream=None, main_start=None,
                                  main_stop=None):
    """Device entry point with events around the dominant kernel.

    main_start / main_stop are torch.cuda.Event objects (recorded at least once
    before, so that their handles exist) or None.  Returns (launches, route).
    """
    nd, B, C_in, C_out, I, K = _problem_from_tensors(x, w, groups)
    ax = _Axes(nd, I, K, stride, pad_lo, pad_hi, dilation, output_padding)
    dev = _same_device(x, w, bias, y, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    n = ctypes.c_int(0)
    r = ctypes.c_int(-1)
    ev = lambda e: None if e is None else e.cuda_event
    with torch.cuda.device(dev):
        s = _stream_handle(stream, dev)
        rc = lib().ct_conv_transpose_nd_profiled(
            _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(workspace), ws_bytes,
            *_shape_args(B, C_in, C_out, ax, groups, dtype_code(x.dtype)), int(route), s,
            ev(main_start), ev(main_stop), ctypes.byref(n), ctypes.byref(r))
    _check(rc)
    return int(n.value), int(r.value)


def ct_conv_transpose_nd_host(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                              y: torch.Tensor, stride=None, pad_lo=None, pad_hi=None,
                              dilation=None, output_padding=None, groups: int = 1,
                              stream=None) -> None:
    """Run the host-buffer entry point on CPU tensors (pinned is fastest)."""
    nd, B, C_in, C_out, I, K = _problem_from_tensors(x, w, groups)
    if bias is not None and tuple(bias.shape) != (C_out,):
        raise CtError(CT_ERR_BIAS, f"bias must have shape [{C_out}], got {tuple(bias.shape)}")
    ax = _Axes(nd, I, K, stride, pad_lo, pad_hi, dilation, output_padding)
    s = _stream_handle(stream, None)
    _check(lib().ct_conv_transpose_nd_host(
        _ptr(x), _ptr(w), _ptr(bias), _ptr(y),
        *_shape_args(B, C_in, C_out, ax, groups, dtype_code(x.dtype)), s))


def ct_conv_transpose_nd_noalloc(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                                 y: torch.Tensor, stride=None, pad_lo=None, pad_hi=None,
                                 dilation=None, output_padding=None, groups: int = 1,
                                 stream=None) -> None:
    """The entry point that allocates no device memory (for callers that may
    not call cudaMalloc where they run the convolution).  It uses the
    library's fixed static scratch; calls that overlap on the GPU race on it."""
    nd, B, C_in, C_out, I, K = _problem_from_tensors(x, w, groups)
    if bias is not None and tuple(bias.shape) != (C_out,):
        raise CtError(CT_ERR_BIAS, f"bias must have shape [{C_out}], got {tuple(bias.shape)}")
    ax = _Axes(nd, I, K, stride, pad_lo, pad_hi, dilation, output_padding)
    dev = _same_device(x, w, bias, y)
    with torch.cuda.device(dev):
        s = _stream_handle(stream, dev)
        rc = lib().ct_conv_transpose_nd_noalloc(
            _ptr(x), _ptr(w), _ptr(bias), _ptr(y),
            *_shape_args(B, C_in, C_out, ax, groups, dtype_code(x.dtype)), s)
    _check(rc)


def ct_host_buffers_release() -> None:
    """Return the device memory the host-buffer entry point keeps in its pool."""
    _check(lib().ct_host_buffers_release())


# Default limit of each bounded device-side wait (CT_WAIT_LIMIT_DEFAULT_NS).
CT_WAIT_LIMIT_DEFAULT_NS = 2_000_000_000


def ct_set_wait_limit_ns(ns: int) -> int:
    """Set the limit of every bounded device-side wait in later launches
    (process-wide; 0 = every wait gives up at once); returns the previous one."""
    return int(lib().ct_set_wait_limit_ns(int(ns)))


def ct_device_status(clear: bool = True):
    """(status, code) of the device-side error word; synchronises the device."""
    code = ctypes.c_uint(0)
    rc = lib().ct_device_status(1 if clear else 0, ctypes.byref(code))
    return rc, int(code.value)


def _attrs(nd, stride, padding, pad_lo, pad_hi, dilation, output_padding):
    def vec(v, default):
        if v is None:
            v = default
        if isinstance(v, int):
            v = [v] * nd
        return [int(a) for a in v]
    pl = vec(pad_lo if pad_lo is not None else padding, 0)
    ph = vec(pad_hi if pad_hi is not None else padding, 0)
    return vec(stride, 1), pl, ph, vec(dilation, 1), vec(output_padding, 0)


def conv_transpose(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                   stride=1, padding=0, pad_lo=None, pad_hi=None, dilation=1, output_padding=0,
                   groups: int = 1, route: int = CT_ROUTE_AUTO,
                   workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Allocate y with the library's output shape and run the device entry point."""
    nd, B, C_in, C_out, I, K = _problem_from_tensors(x, w, groups)
    s, pl, ph, d, op = _attrs(nd, stride, padding, pad_lo, pad_hi, dilation, output_padding)
    O = ct_conv_transpose_out_shape(I, K, s, pl, ph, d, op)
    y = torch.empty((B, C_out) + O, dtype=x.dtype, device=x.device)
    ct_conv_transpose_nd(x, w, bias, y, workspace, s, pl, ph, d, op, groups, route)
    return y


def ct_conv_transpose_backward_workspace_bytes(B, C_in, C_out, in_spatial, k, stride=None,
                                               pad_lo=None, pad_hi=None, dilation=None,
                                               output_padding=None, groups=1,
                                               dtype=CT_F32) -> int:
    ax = _Axes(len(in_spatial), in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding)
    n = ctypes.c_size_t(0)
    _check(lib().ct_conv_transpose_backward_workspace_bytes(
        *_shape_args(B, C_in, C_out, ax, groups, dtype), ctypes.byref(n)))
    return int(n.value)


def ct_conv_transpose_backward_nd(x: torch.Tensor, w: torch.Tensor, dy: torch.Tensor,
                                  dx: Optional[torch.Tensor] = None,
                                  dw: Optional[torch.Tensor] = None,
                                  db: Optional[torch.Tensor] = None,
                                  workspace: Optional[torch.Tensor] = None, stride=None,
                                  pad_lo=None, pad_hi=None, dilation=None, output_padding=None,
                                  groups: int = 1, stream=None) -> None:
    """Run the backward entry point on torch CUDA tensors; dx, dw and db (any
    may be None) are overwritten."""
    nd, B, C_in, C_out, I, K = _problem_from_tensors(x, w, groups)
    ax = _Axes(nd, I, K, stride, pad_lo, pad_hi, dilation, output_padding)
    nws = workspace.numel() * workspace.element_size() if workspace is not None else 0
    dev = _same_device(x, w, dy, dx, dw, db, workspace)
    with torch.cuda.device(dev):
        s = _stream_handle(stream, dev)
        rc = lib().ct_conv_transpose_backward_nd(
            _ptr(x), _ptr(w), _ptr(dy), _ptr(dx), _ptr(dw), _ptr(db), _ptr(workspace), nws,
            *_shape_args(B, C_in, C_out, ax, groups, dtype_code(dy.dtype)), s)
    _check(rc)


def conv_transpose_backward(x: torch.Tensor, w: torch.Tensor, dy: torch.Tensor, stride=1,
                            padding=0, pad_lo=None, pad_hi=None, dilation=1, output_padding=0,
                            groups: int = 1, need=("dx", "dw", "db")):
    """Allocate and return (dx, dw, db) for upstream gradient dy; entries not
    in `need` are None."""
    nd, B, C_in, C_out, I, K = _problem_from_tensors(x, w, groups)
    s, pl, ph, d, op = _attrs(nd, stride, padding, pad_lo, pad_hi, dilation, output_padding)
    dx = torch.empty_like(x) if "dx" in need else None
    dw = torch.empty_like(w) if "dw" in need else None
    db = torch.empty((C_out,), dtype=dy.dtype, device=dy.device) if "db" in need else None
    ct_conv_transpose_backward_nd(x, w, dy, dx, dw, db, None, s, pl, ph, d, op, groups)
    return dx, dw, db


class ConvTransposeFunction(torch.autograd.Function):
    """torch.autograd binding: forward and backward both run in libct.so."""

    @staticmethod
    def forward(ctx, x, w, bias, stride, padding, pad_lo, pad_hi, dilation, output_padding,
                groups):
        ctx.save_for_backward(x, w)
        ctx.attrs = (stride, padding, pad_lo, pad_hi, dilation, output_padding, groups)
        ctx.has_bias = bias is not None
        return conv_transpose(x, w, bias, stride, padding, pad_lo, pad_hi, dilation,
                              output_padding, groups)

    @staticmethod
    def backward(ctx, dy):
        x, w = ctx.saved_tensors
        stride, padding, pad_lo, pad_hi, dilation, output_padding, groups = ctx.attrs
        need = tuple(n for n, flag in (("dx", ctx.needs_input_grad[0]),
                                       ("dw", ctx.needs_input_grad[1]),
                                       ("db", ctx.needs_input_grad[2] and ctx.has_bias)) if flag)
        dx, dw, db = conv_transpose_backward(x, w, dy.contiguous(), stride, padding, pad_lo,
                                             pad_hi, dilation, output_padding, groups, need)
        return (dx, dw, db, None, None, None, None, None, None, None)


def conv_transpose_autograd(x, w, bias=None, stride=1, padding=0, pad_lo=None, pad_hi=None,
                            dilation=1, output_padding=0, groups=1):
    """conv_transpose that records itself for torch.autograd."""
    return ConvTransposeFunction.apply(x, w, bias, stride, padding, pad_lo, pad_hi, dilation,
                                       output_padding, groups)


def _problem_ex(x, w, groups, w_layout):
    """(nd, B, C_in, C_out, I, K) for a weight in any ct_weight_layout."""
    if w_layout == CT_W_TORCH:
        return _problem_from_tensors(x, w, groups)
    nd = x.dim() - 2
    if nd < 1 or w.dim() != x.dim():
        raise CtError(CT_ERR_RANK, "x must be [B, C_in, *spatial] and w [*k, C_in, C_out] "
                                   "or [*k, C_out, C_in]")
    C_out = w.shape[-1] if w_layout == CT_W_KDHW_CI_CO else w.shape[-2]
    return nd, x.shape[0], x.shape[1], C_out, tuple(x.shape[2:]), tuple(w.shape[:nd])


def ct_conv_transpose_ex_workspace_bytes(B, C_in, C_out, in_spatial, k, stride=None, pad_lo=None,
                                         pad_hi=None, dilation=None, output_padding=None,
                                         groups=1, dtype=CT_F32, w_layout=CT_W_TORCH,
                                         taps_flipped=0) -> int:
    ax = _Axes(len(in_spatial), in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding)
    n = ctypes.c_size_t(0)
    _check(lib().ct_conv_transpose_ex_workspace_bytes(
        *_shape_args(B, C_in, C_out, ax, groups, dtype), int(w_layout), int(taps_flipped),
        ctypes.byref(n)))
    return int(n.value)


def ct_conv_transpose_nd_ex(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                            y: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                            stride=None, pad_lo=None, pad_hi=None, dilation=None,
                            output_padding=None, groups: int = 1, w_layout: int = CT_W_TORCH,
                            taps_flipped: int = 0, activation=CT_ACT_NONE,
                            activation_alpha: float = 0.01, stream=None) -> None:
    """Run the extended entry point (weight layout, flipped taps, fused
    activation) on torch CUDA tensors; y is overwritten."""
    nd, B, C_in, C_out, I, K = _problem_ex(x, w, groups, w_layout)
    act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
    ax = _Axes(nd, I, K, stride, pad_lo, pad_hi, dilation, output_padding)
    nws = workspace.numel() * workspace.element_size() if workspace is not None else 0
    dev = _same_device(x, w, bias, y, workspace)
    with torch.cuda.device(dev):
        s = _stream_handle(stream, dev)
        rc = lib().ct_conv_transpose_nd_ex(
            _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(workspace), nws,
            *_shape_args(B, C_in, C_out, ax, groups, dtype_code(x.dtype)), int(w_layout),
            int(taps_flipped), act, float(activation_alpha), s)
    _check(rc)

