"""GPU parity of the CUDA-core routes: the fp32 SIMT phase GEMM and the
grouped/depthwise stride-phase gather, each forced onto its route and
compared with the fp64 oracle.  Shapes cover ragged tiles (channels and
positions not multiples of the 128 x 128 GEMM tile or the 8-row blocks),
strides 1..8, dilation, asymmetric pads, output_padding, phases without
taps, 1-D/2-D/3-D, depthwise, and the three dtypes on the grouped route.
"""
import pytest
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import assert_close, run, supported_routes

pytestmark = pytest.mark.gpu

P = synth.problem
SIMT_CASES = [
    P("simt_1d_c1_like", 2, 96, 72, (300,), 8, stride=4, pad=2, seed=301),
    P("simt_1d_s1", 2, 40, 130, (257,), 5, stride=1, pad=2, seed=302),
    P("simt_1d_s3_dil", 1, 33, 48, (101,), 4, stride=3, pad_lo=1, pad_hi=3, dilation=2,
      output_padding=2, seed=303),
    P("simt_1d_s8", 1, 64, 64, (64,), 16, stride=8, pad=4, seed=304),
    P("simt_2d", 2, 64, 40, (13, 21), 4, stride=2, pad=1, seed=305),
    P("simt_2d_empty_phases", 1, 32, 32, (6, 7), 2, stride=5, output_padding=(4, 3), seed=306),
    P("simt_3d", 1, 32, 48, (3, 7, 9), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
      seed=307),
    P("simt_no_bias", 3, 48, 64, (77,), 3, stride=2, pad=1, bias=False, seed=308),
    P("simt_wide", 1, 128, 260, (150,), 4, stride=2, pad=1, seed=309),
]

GROUPED_CASES = [
    P("grp_c3_like", 2, 64, 64, (20, 23), 3, stride=2, pad=1, dilation=2, output_padding=1,
      groups=8, seed=401),
    P("grp_depthwise", 2, 24, 24, (17, 15), 4, stride=2, pad=1, groups=24, seed=402),
    P("grp_depthwise_mult", 1, 8, 32, (9, 11), 3, stride=3, pad=1, output_padding=2, groups=8,
      seed=403),
    P("grp_s1", 2, 32, 32, (12, 40), 5, stride=1, pad=2, groups=4, seed=404),
    P("grp_s4_1d", 2, 16, 32, (70,), 8, stride=4, pad=2, groups=2, seed=405),
    P("grp_3d", 1, 16, 16, (3, 6, 7), 3, stride=2, pad=1, output_padding=1, groups=4, seed=406),
    P("grp_bf16", 2, 64, 64, (20, 23), 3, stride=2, pad=1, dilation=2, output_padding=1,
      groups=32, dtype="bf16", seed=407),
    P("grp_f16", 1, 32, 48, (10, 9), 4, stride=2, pad_lo=2, pad_hi=0, groups=4, dtype="f16",
      seed=408),
    P("grp_small_dense", 1, 4, 3, (8, 8), 3, stride=2, pad=1, output_padding=1, seed=409),
    P("grp_empty_phases", 1, 8, 8, (6, 5), 2, stride=4, output_padding=(3, 2), groups=2,
      seed=410),
]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transposed_convolution_convtranspose1_gb300 import _build
    _build.build_library()
    ct.lib()
    yield


def _check(p, route):
    assert route in supported_routes(p), p.name
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    y = run(p, x, w, b, route=route)
    torch.cuda.synchronize()
    assert_close(p, y, ref, f"route {route}")


@pytest.mark.parametrize("p", SIMT_CASES, ids=lambda p: p.name)
def test_simt_route_matches_oracle(p):
    _check(p, ct.CT_ROUTE_SIMT_GEMM)


@pytest.mark.parametrize("p", GROUPED_CASES, ids=lambda p: p.name)
def test_grouped_route_matches_oracle(p):
    _check(p, ct.CT_ROUTE_GROUPED)


def test_auto_routes_of_the_workloads():
    want = {0: ct.CT_ROUTE_GROUPED, 1: ct.CT_ROUTE_TC32_GEMM, 2: ct.CT_ROUTE_TC_GEMM,
            3: ct.CT_ROUTE_GROUPED, 4: ct.CT_ROUTE_TC_GEMM}
    for i, r in want.items():
        p = synth.workload(i)
        got = ct.ct_conv_transpose_route(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride,
                                         p.pad_lo, p.pad_hi, p.dilation, p.output_padding,
                                         p.groups, ct.dtype_code(p.torch_dtype))
        assert got == r, (p.name, got, r)


def test_dominant_kernel_of_the_workloads():
    """ct_conv_transpose_kernel names the kernel each workload's time goes
    to: the small 2-D case (4 input channels per group) takes the staged
    grouped kernel, the grouped workload (8 per group, fp32, width 56) the
    warp-pipeline one; a bf16 grouped problem stays on the staged kernel."""
    want = {0: "grouped_staged_kernel", 1: "tc32_phase_gemm", 2: "tc_phase_gemm",
            3: "grouped_warp_kernel", 4: "tc_phase_gemm"}
    for i, name in want.items():
        p = synth.workload(i)
        got = ct.ct_conv_transpose_kernel(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride,
                                          p.pad_lo, p.pad_hi, p.dilation, p.output_padding,
                                          p.groups, ct.dtype_code(p.torch_dtype))
        assert got == name, (p.name, got, name)
    p = synth.workload(3).replace(dtype="bf16")
    got = ct.ct_conv_transpose_kernel(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo,
                                      p.pad_hi, p.dilation, p.output_padding, p.groups,
                                      ct.dtype_code(p.torch_dtype))
    assert got == "grouped_staged_kernel"
    empty = ct.ct_conv_transpose_kernel(0, 4, 6, (5,), (3,), (2,))
    assert empty == ""
