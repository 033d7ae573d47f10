"""Host-side checks of the C ABI (no GPU needed, no compute calls).

- libct.so builds, loads and exports every function include/ct.h declares;
- ct_conv_transpose_out_shape agrees with the golden shapes and the oracle;
- every invalid argument is rejected with its status code before any launch.
"""
import ctypes
import json
import os
import re

import numpy as np
import pytest
import torch

import oracle
from transposed_convolution_convtranspose1_gb300 import _build
from transposed_convolution_convtranspose1_gb300 import ct as ctb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ct.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "out_shapes.json")


@pytest.fixture(scope="module")
def lib():
    _build.build_library()
    return ctb.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ct_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ct_conv_transpose_nd", "ct_conv_transpose_out_shape",
                 "ct_conv_transpose_workspace_bytes", "ct_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ct.h but not exported"
    assert set(ctb.EXPORTS) <= set(names)


def test_version_and_status_strings(lib):
    assert ctb.ct_version() >= 100
    assert ctb.ct_status_string(0) == "CT_OK"
    assert ctb.ct_status_string(7) == "CT_ERR_DTYPE"


def test_out_shape_golden(lib):
    for c in json.load(open(GOLDEN))["cases"]:
        got = ctb.ct_conv_transpose_out_shape(c["x"][2:], c["w"][2:], c["stride"], c["pad_lo"],
                                              c["pad_hi"], c["dilation"], c["output_padding"])
        assert (c["x"][0], c["w"][1] * c["groups"]) + got == tuple(c["y"]), c["source"]


def test_out_shape_agrees_with_oracle_on_a_grid(lib):
    r = np.random.default_rng(5)
    for _ in range(300):
        nd = int(r.integers(1, 4))
        I = [int(r.integers(0, 40)) for _ in range(nd)]
        k = [int(r.integers(1, 8)) for _ in range(nd)]
        s = [int(r.integers(1, 6)) for _ in range(nd)]
        d = [int(r.integers(1, 4)) for _ in range(nd)]
        pl = [int(r.integers(0, 6)) for _ in range(nd)]
        ph = [int(r.integers(0, 6)) for _ in range(nd)]
        op = [int(r.integers(0, max(a, b))) for a, b in zip(s, d)]
        try:
            want = oracle.out_shape(I, k, s, pl, ph, d, op)
        except ValueError:
            want = None
        if want is None:
            with pytest.raises(ctb.CtError) as e:
                ctb.ct_conv_transpose_out_shape(I, k, s, pl, ph, d, op)
            assert e.value.status in (ctb.CT_ERR_SHAPE,)
        else:
            assert ctb.ct_conv_transpose_out_shape(I, k, s, pl, ph, d, op) == want


def _call(lib, **kw):
    """ct_conv_transpose_nd with fake (never dereferenced) device pointers."""
    p = dict(x=256, w=512, bias=None, y=1024, ws=None, ws_bytes=0, nd=2, B=1, C_in=4, C_out=6,
             I=[5, 5], k=[3, 3], s=[2, 2], pl=[1, 1], ph=[1, 1], d=[1, 1], op=[0, 0], groups=2,
             dtype=ctb.CT_F32)
    p.update(kw)
    ax = ctb._Axes(len(p["I"]), p["I"], p["k"], p["s"], p["pl"], p["ph"], p["d"], p["op"])
    ax.nd = p["nd"]
    return lib.ct_conv_transpose_nd(p["x"], p["w"], p["bias"], p["y"], p["ws"], p["ws_bytes"],
                                    *ctb._shape_args(p["B"], p["C_in"], p["C_out"], ax,
                                                     p["groups"], p["dtype"]), None)


def test_validation_rejects_before_launch(lib):
    cases = [
        (dict(nd=0, I=[], k=[], s=[], pl=[], ph=[], d=[], op=[]), ctb.CT_ERR_RANK),
        (dict(nd=4, I=[2] * 4, k=[1] * 4, s=[1] * 4, pl=[0] * 4, ph=[0] * 4, d=[1] * 4,
              op=[0] * 4), ctb.CT_ERR_RANK),
        (dict(x=None), ctb.CT_ERR_NULL),
        (dict(w=None), ctb.CT_ERR_NULL),
        (dict(y=None), ctb.CT_ERR_NULL),
        (dict(I=[-1, 5]), ctb.CT_ERR_SHAPE),
        (dict(B=-1), ctb.CT_ERR_SHAPE),
        (dict(k=[0, 3]), ctb.CT_ERR_PARAM),
        (dict(s=[0, 2]), ctb.CT_ERR_PARAM),
        (dict(d=[1, 0]), ctb.CT_ERR_PARAM),
        (dict(pl=[-1, 1]), ctb.CT_ERR_PARAM),
        (dict(op=[2, 0]), ctb.CT_ERR_PARAM),          # op >= max(stride, dilation)
        (dict(op=[-1, 0]), ctb.CT_ERR_PARAM),
        (dict(s=[1, 1], pl=[4, 4], ph=[4, 4]), ctb.CT_ERR_SHAPE),  # O = 4-8+2+1 = -1
        (dict(groups=0), ctb.CT_ERR_GROUPS),
        (dict(groups=3), ctb.CT_ERR_GROUPS),          # 3 does not divide C_in=4
        (dict(C_out=5), ctb.CT_ERR_GROUPS),           # groups=2 does not divide C_out=5
        (dict(dtype=3), ctb.CT_ERR_DTYPE),
        (dict(dtype=-1), ctb.CT_ERR_DTYPE),
        (dict(x=258), ctb.CT_ERR_ALIGN),              # fp32 pointer not 4-byte aligned
        (dict(k=[33, 3]), ctb.CT_ERR_TOO_LARGE),
    ]
    for kw, want in cases:
        rc = _call(lib, **kw)
        assert rc == want, (kw, rc, ctb.ct_last_error())
        assert ctb.ct_last_error()


def test_op_bound_uses_max_of_stride_and_dilation(lib):
    # stride 1, dilation 3: op = 2 is legal in validation; the shape is then fine.
    out = ctb.ct_conv_transpose_out_shape([4], [3], [1], [0], [0], [3], [2])
    assert out == ((4 - 1) * 1 + 3 * 2 + 2 + 1,)
    with pytest.raises(ctb.CtError) as e:
        ctb.ct_conv_transpose_out_shape([4], [3], [1], [0], [0], [3], [3])
    assert e.value.status == ctb.CT_ERR_PARAM


def test_binding_rejects_integer_dtype_through_the_abi(lib):
    x = torch.zeros((1, 2, 3), dtype=torch.int32)
    w = torch.zeros((2, 2, 2), dtype=torch.int32)
    y = torch.zeros((1, 2, 4), dtype=torch.int32)
    with pytest.raises(ctb.CtError) as e:
        ctb.ct_conv_transpose_nd(x, w, None, y, stream=0)
    assert e.value.status == ctb.CT_ERR_DTYPE


def test_binding_rejects_bad_bias_shape(lib):
    x = torch.zeros((1, 2, 3))
    w = torch.zeros((2, 2, 2))
    y = torch.zeros((1, 2, 4))
    with pytest.raises(ctb.CtError) as e:
        ctb.ct_conv_transpose_nd(x, w, torch.zeros(3), y, stream=0)
    assert e.value.status == ctb.CT_ERR_BIAS


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(ctb, "_lib_handle", None)
    monkeypatch.setattr(ctb, "LIB_PATH", os.path.join(ROOT, "no_such_libct.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        ctb.lib()


def test_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "transposed_convolution_convtranspose1_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, flags=re.M), f
                assert "ct_oracle" not in text, f


def test_extended_call_validates_its_options_before_launch(lib):
    """ct_conv_transpose_nd_ex (the C entry point): unknown layout, flag or
    activation -> CT_ERR_PARAM; the NKI layouts with groups != 1 ->
    CT_ERR_GROUPS; all before any device work (the buffer pointers are never
    touched: stand-in host addresses)."""
    import ctypes
    buf = (ctypes.c_float * 64)()
    ptr = ctypes.cast(buf, ctypes.c_void_p).value
    ax = ctb._Axes(1, (3,), (2,), None, None, None, None, None)

    def call(w_layout=ctb.CT_W_KDHW_CI_CO, taps_flipped=0, activation=0, groups=1):
        return lib.ct_conv_transpose_nd_ex(
            ptr, ptr, None, ptr, None, 0, *ctb._shape_args(1, 4, 6, ax, groups, ctb.CT_F32),
            int(w_layout), int(taps_flipped), int(activation), 0.01, None)

    for kw in (dict(w_layout=3), dict(taps_flipped=2), dict(activation=7), dict(activation=-1)):
        assert call(**kw) == ctb.CT_ERR_PARAM, kw
    assert call(groups=2) == ctb.CT_ERR_GROUPS   # [k, C_in, C_out] with groups 2
    # workspace of a flipped PyTorch-layout weight: at least the weight's bytes
    n = ctb.ct_conv_transpose_ex_workspace_bytes(1, 4, 6, [3], [2], [1], [0], [0], [1], [0],
                                                 1, ctb.CT_F32, ctb.CT_W_TORCH, 1)
    assert n >= 4 * 6 * 2 * 4


def test_binding_wants_device_tensors_on_one_device(lib):
    """The device-buffer bindings refuse host tensors (a kernel would read host
    memory) before calling the library."""
    x = torch.zeros((1, 2, 3))
    w = torch.zeros((2, 2, 2))
    y = torch.zeros((1, 2, 4))
    with pytest.raises(ctb.CtError, match="device tensors expected") as e:
        ctb.ct_conv_transpose_nd(x, w, None, y, stride=1)
    assert e.value.status == ctb.CT_ERR_PARAM


def test_kernel_query_validates_before_any_device_work(lib):
    """ct_conv_transpose_kernel rejects what ct_conv_transpose_nd rejects (a
    bad output size, output_padding at the stride, groups not dividing C_in,
    an integer dtype) and a NULL result pointer, all on the host."""
    import ctypes
    q = ctb.ct_conv_transpose_kernel
    with pytest.raises(ctb.CtError) as e:
        q(1, 4, 6, (1,), (1,), (1,), (1,), (1,))          # output size 1 - 2 < 1
    assert e.value.status == ctb.CT_ERR_SHAPE
    with pytest.raises(ctb.CtError) as e:
        q(1, 4, 6, (5,), (3,), (2,), output_padding=(2,))
    assert e.value.status == ctb.CT_ERR_PARAM
    with pytest.raises(ctb.CtError) as e:
        q(1, 6, 6, (5,), (3,), (2,), groups=4)
    assert e.value.status == ctb.CT_ERR_GROUPS
    with pytest.raises(ctb.CtError) as e:
        q(1, 4, 6, (5,), (3,), (2,), dtype=7)
    assert e.value.status == ctb.CT_ERR_DTYPE
    ax = ctb._Axes(1, (5,), (3,), (2,), None, None, None, None)
    rc = lib.ct_conv_transpose_kernel(*ctb._shape_args(1, 4, 6, ax, 1, ctb.CT_F32),
                                      ctypes.cast(None, ctypes.POINTER(ctypes.c_char_p)))
    assert rc == ctb.CT_ERR_NULL


def test_backward_kernel_query_validates_on_the_host(lib):
    """ct_conv_transpose_backward_kernels rejects a bad shape, groups that do
    not divide the channels, an integer dtype and NULL result pointers, and
    on a problem the backward call accepts it names one kernel per gradient
    from the two each gradient has (the tensor-core dx needs an sm_103 device,
    which this host check does not assume)."""
    import ctypes
    q = ctb.ct_conv_transpose_backward_kernels
    with pytest.raises(ctb.CtError) as e:
        q(1, 4, 6, (1,), (1,), (1,), (1,), (1,))
    assert e.value.status == ctb.CT_ERR_SHAPE
    with pytest.raises(ctb.CtError) as e:
        q(1, 6, 6, (5,), (3,), (2,), groups=4)
    assert e.value.status == ctb.CT_ERR_GROUPS
    with pytest.raises(ctb.CtError) as e:
        q(1, 4, 6, (5,), (3,), (2,), dtype=7)
    assert e.value.status == ctb.CT_ERR_DTYPE
    ax = ctb._Axes(1, (5,), (3,), (2,), None, None, None, None)
    null = ctypes.cast(None, ctypes.POINTER(ctypes.c_char_p))
    rc = lib.ct_conv_transpose_backward_kernels(*ctb._shape_args(1, 4, 6, ax, 1, ctb.CT_F32), null, null)
    assert rc == ctb.CT_ERR_NULL
    dx, dw = q(2, 64, 32, (9, 9), (3, 3), (2, 2), dtype=ctb.CT_BF16)
    assert dx in ("tc_phase_gemm", "bwd_dx_kernel") and dw in ("tc_dw_gemm", "bwd_dw_kernel")
    assert q(2, 64, 32, (9, 9), (3, 3), (2, 2))[0] in ("tc32_phase_gemm", "bwd_dx_kernel")
    assert q(2, 16, 16, (9, 9), (3, 3), (2, 2), groups=2)[1] == "bwd_dw_grouped_kernel"
    assert q(0, 16, 16, (9, 9), (3, 3), (2, 2))[0] == ""
