"""GPU tests of ct_conv_transpose_nd_ex: the NKI page's conv3d_transpose
options (weight layouts KDHW_CI_CO / KDHW_CO_CI, caller-flipped taps, an
activation applied after the convolution).

- Activations: every activation on every route a problem supports, against
  oracle.activation of the fp64 oracle's output.  Bound: the dtype's
  tolerance times max(max|act(y)|, max|y|) -- an activation's slope is at most
  about 1.13 (gelu), so the pre-activation error scale carries over.
- Layouts and flipped taps: the same weights rewritten into each layout (by
  numpy in the test) give y bit for bit equal to the plain call's.
"""
import numpy as np
import pytest
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import TOL

pytestmark = pytest.mark.gpu

P = synth.problem


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transposed_convolution_convtranspose1_gb300 import _build
    _build.build_library()
    ct.lib()
    ct.ct_device_status(clear=True)
    yield
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.CT_OK, f"device error word set: {code:#x}"


def _out(p):
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    return torch.empty((p.B, p.C_out) + tuple(O), dtype=p.torch_dtype, device="cuda")


def _run_ex(p, x, w, b, **kw):
    y = _out(p)
    ct.ct_conv_transpose_nd_ex(x.cuda(), w.cuda(), None if b is None else b.cuda(), y, None,
                               p.stride, p.pad_lo, p.pad_hi, p.dilation, p.output_padding,
                               p.groups, **kw)
    torch.cuda.synchronize()
    return y


ACT_PROBLEMS = [
    synth.workload(0),                                               # grouped route
    P("act_tc32", 2, 64, 40, (37,), 8, stride=4, pad=2, seed=601),   # TF32 route
    P("act_bf16", 2, 64, 48, (9, 11), 4, stride=2, pad=1, dtype="bf16", seed=602),  # tcgen05
    P("act_f16_3d", 1, 32, 24, (3, 5, 6), 3, stride=(1, 2, 2), pad=1,
      output_padding=(0, 1, 1), dtype="f16", seed=603),
    P("act_gather", 1, 3, 40, (7, 5), 3, stride=3, dilation=2, pad=1, seed=604),  # generic
    P("act_simt_like", 1, 40, 36, (30,), 12, stride=1, pad=3, seed=605),  # 12 taps: SIMT
    P("act_grouped_bf16", 2, 16, 16, (6, 7), 3, stride=2, groups=4, pad=1, dtype="bf16",
      seed=606),
    P("act_bias_only", 1, 4, 6, (0, 5), 3, stride=2, seed=607),       # bias fill
]


@pytest.mark.parametrize("act", ["relu", "leaky_relu", "silu", "gelu", "tanh", "sigmoid"])
@pytest.mark.parametrize("p", ACT_PROBLEMS, ids=lambda p: p.name)
def test_activation_matches_oracle(p, act):
    x, w, b = synth.make_inputs(p)
    y = _run_ex(p, x, w, b, activation=act, activation_alpha=0.07)
    pre = oracle.conv_transpose(x, w, b, **p.attrs())
    ref = oracle.activation(pre, act, 0.07)
    got = y.to(torch.float64).cpu().numpy()
    scale = max(float(np.max(np.abs(ref))) if ref.size else 0.0,
                float(np.max(np.abs(pre))) if pre.size else 0.0)
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= TOL[p.dtype] * scale, f"{p.name} {act}: {err:.3e} > {TOL[p.dtype]} * {scale:.3e}"


def test_activation_reaches_every_route_epilogue():
    """The extended call takes the automatic route, so each route's epilogue
    is reached through a problem the choice sends to it: the problems above
    cover grouped, TF32, tcgen05, SIMT (12 taps per phase are beyond the
    TF32 route's 8), generic gather and bias fill."""
    routes = set()
    for p in ACT_PROBLEMS:
        routes.add(ct.ct_conv_transpose_route(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride,
                                              p.pad_lo, p.pad_hi, p.dilation, p.output_padding,
                                              p.groups, ct.dtype_code(p.torch_dtype)))
    for r in (ct.CT_ROUTE_GROUPED, ct.CT_ROUTE_TC32_GEMM, ct.CT_ROUTE_TC_GEMM,
              ct.CT_ROUTE_SIMT_GEMM, ct.CT_ROUTE_GATHER, ct.CT_ROUTE_BIAS_FILL):
        assert r in routes, (r, routes)


def _to_layout(w, nd, layout, flipped):
    """PyTorch-layout weights [C_in, C_out, k...] as the NKI page stores them."""
    a = w.clone()
    if flipped:
        a = torch.flip(a, dims=list(range(2, 2 + nd)))
    if layout == ct.CT_W_TORCH:
        return a.contiguous()
    perm = list(range(2, 2 + nd)) + ([0, 1] if layout == ct.CT_W_KDHW_CI_CO else [1, 0])
    return a.permute(*perm).contiguous()


LAYOUT_PROBLEMS = [
    P("lay_1d_f32", 2, 40, 36, (33,), 8, stride=4, pad=2, seed=611),
    P("lay_2d_bf16", 1, 64, 64, (7, 9), 3, stride=2, pad=1, output_padding=1, dtype="bf16",
      seed=612),
    P("lay_3d_f32", 1, 8, 12, (3, 4, 5), (3, 2, 3), stride=(1, 2, 2), pad=(1, 0, 1), seed=613),
]


@pytest.mark.parametrize("layout,flipped", [(0, 1), (1, 0), (1, 1), (2, 0), (2, 1)])
@pytest.mark.parametrize("p", LAYOUT_PROBLEMS, ids=lambda p: p.name)
def test_weight_layouts_give_the_plain_result(p, layout, flipped):
    x, w, b = synth.make_inputs(p)
    y0 = _out(p)
    ct.ct_conv_transpose_nd(x.cuda(), w.cuda(), b.cuda(), y0, None, p.stride, p.pad_lo, p.pad_hi,
                            p.dilation, p.output_padding, p.groups)
    wl = _to_layout(w, len(p.spatial), layout, flipped)
    y1 = _run_ex(p, x, wl, b, w_layout=layout, taps_flipped=flipped)
    assert torch.equal(y0, y1)


def test_caller_workspace_for_a_converted_weight():
    p = LAYOUT_PROBLEMS[0]
    x, w, b = synth.make_inputs(p)
    n = ct.ct_conv_transpose_ex_workspace_bytes(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride,
                                                p.pad_lo, p.pad_hi, p.dilation, p.output_padding,
                                                p.groups, ct.dtype_code(p.torch_dtype),
                                                ct.CT_W_KDHW_CO_CI, 1)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    y0, y1 = _out(p), _out(p)
    ct.ct_conv_transpose_nd(x.cuda(), w.cuda(), b.cuda(), y0, None, p.stride, p.pad_lo, p.pad_hi,
                            p.dilation, p.output_padding, p.groups)
    ct.ct_conv_transpose_nd_ex(x.cuda(), _to_layout(w, 1, 2, 1).cuda(), b.cuda(), y1, ws,
                               p.stride, p.pad_lo, p.pad_hi, p.dilation, p.output_padding,
                               p.groups, w_layout=2, taps_flipped=1, activation="relu")
    torch.cuda.synchronize()
    assert torch.equal(torch.relu(y0), y1)
    with pytest.raises(ct.CtError) as e:
        ct.ct_conv_transpose_nd_ex(x.cuda(), _to_layout(w, 1, 2, 1).cuda(), b.cuda(), y1,
                                   ws[: n // 2], p.stride, p.pad_lo, p.pad_hi, p.dilation,
                                   p.output_padding, p.groups, w_layout=2, taps_flipped=1)
    assert e.value.status == ct.ct.CT_ERR_WORKSPACE
