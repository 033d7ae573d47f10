"""GPU parity of the tcgen05 route (bf16/fp16 stride-phase implicit GEMM).

Shapes are chosen to hit the route's corners: tiles of 8..128 positions per
row (W extents from tiny to > 128), several rows per tile, ragged tails on
every axis, C_in not a multiple of the 64-channel k-block, C_out not a
multiple of 16 and larger than one channel tile, strides 1..4 (1..4
accumulators per tile), phases without taps, 1-D/2-D/3-D, dilation,
asymmetric pads and output_padding.  Every case is forced onto the route and
compared with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import assert_close, run, supported_routes

pytestmark = pytest.mark.gpu

P = synth.problem
CASES = [
    P("tc_2d_basic", 2, 64, 64, (16, 16), 4, stride=2, pad=1, dtype="bf16", seed=201),
    P("tc_2d_f16", 2, 64, 64, (16, 16), 4, stride=2, pad=1, dtype="f16", seed=202),
    P("tc_ragged_c", 3, 72, 40, (13, 19), 3, stride=2, pad_lo=(1, 0), pad_hi=(0, 2),
      output_padding=(1, 1), dtype="bf16", seed=203),
    P("tc_wide_w", 1, 64, 48, (5, 150), (3, 4), stride=(1, 2), pad=1, dtype="bf16", seed=204),
    P("tc_tiny_w", 2, 32, 32, (37, 3), 3, stride=2, pad=0, dtype="bf16", seed=205),
    P("tc_stride1", 2, 96, 200, (11, 17), 3, stride=1, pad=1, dtype="bf16", seed=206),
    P("tc_stride3", 1, 64, 80, (10, 12), 5, stride=3, pad=2, output_padding=2, dtype="bf16",
      seed=207),
    P("tc_stride4_1d", 2, 128, 64, (300,), 8, stride=4, pad=2, dtype="bf16", seed=208),
    P("tc_two_oc_tiles", 1, 64, 256, (9, 9), 4, stride=2, pad=1, dtype="bf16", seed=209),
    P("tc_3d", 1, 64, 48, (4, 9, 10), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
      dtype="bf16", seed=210),
    P("tc_3d_s2", 1, 32, 32, (3, 5, 7), (2, 3, 3), stride=2, pad=(0, 1, 1), dtype="f16",
      seed=211),
    P("tc_dilated", 2, 64, 32, (12, 12), 3, stride=2, pad=1, dilation=2, output_padding=1,
      dtype="bf16", seed=212),
    P("tc_empty_phases", 1, 64, 32, (7, 8), 2, stride=4, pad=0, output_padding=(3, 2),
      dtype="bf16", seed=213),
    P("tc_no_bias", 2, 64, 64, (8, 8), 2, stride=2, dtype="bf16", bias=False, seed=214),
    P("tc_1x1", 2, 128, 96, (33, 31), 1, dtype="bf16", seed=215),
    P("tc_big_k", 1, 512, 64, (8, 8), 4, stride=2, pad=1, dtype="bf16", seed=216),
]


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


@pytest.mark.parametrize("p", CASES, ids=lambda p: p.name)
def test_tc_route_matches_oracle(p):
    assert ct.CT_ROUTE_TC_GEMM in supported_routes(p), p.name
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    y = run(p, x, w, b, route=ct.CT_ROUTE_TC_GEMM)
    torch.cuda.synchronize()
    assert_close(p, y, ref, "tc route")
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.CT_OK, f"{p.name}: device error word {code:#x}"


@pytest.mark.parametrize("i", [2, 4])
def test_auto_route_is_tc_for_bf16_workloads(i):
    p = synth.workload(i)
    r = ct.ct_conv_transpose_route(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo,
                                   p.pad_hi, p.dilation, p.output_padding, p.groups,
                                   ct.dtype_code(p.torch_dtype))
    assert r == ct.CT_ROUTE_TC_GEMM


def test_tc_route_rejects_grouped_and_fp32():
    p = synth.problem("g2", 1, 64, 64, (8, 8), 3, stride=2, groups=2, dtype="bf16")
    assert ct.CT_ROUTE_TC_GEMM not in supported_routes(p)
    p = synth.problem("f32", 1, 64, 64, (8, 8), 3, stride=2, dtype="f32")
    assert ct.CT_ROUTE_TC_GEMM not in supported_routes(p)


def test_tc_matches_gather_bits_closely():
    """Same inputs through the tensor-core and the gather route: both sum in
    fp32 (in different orders) and round once to bf16, so they differ by at
    most one bf16 ulp of the result plus the fp32 summation-order error,
    bounded here by 1e-5 of the largest output."""
    p = synth.workload(2).replace(B=2, name="c2_b2")
    x, w, b = synth.make_inputs(p)
    yt = run(p, x, w, b, route=ct.CT_ROUTE_TC_GEMM).float()
    yg = run(p, x, w, b, route=ct.CT_ROUTE_GATHER).float()
    torch.cuda.synchronize()
    bound = torch.abs(yg) * 2.0 ** -7 + 1e-5 * float(torch.abs(yg).max())
    assert bool((torch.abs(yt - yg) <= bound).all())


def test_tc_route_with_unaligned_x_and_odd_spatial_size():
    """x starting 2 bytes past a 16-byte boundary and D*H*W not a multiple of
    8 take the layout pass's element-wise path; results must not change."""
    p = synth.problem("tc_unaligned", 2, 64, 32, (7, 9), 3, stride=2, pad=1, dtype="bf16",
                      seed=217)
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    flat = torch.empty(x.numel() + 8, dtype=x.dtype, device="cuda")
    xs = flat[1:1 + x.numel()].view(x.shape)
    xs.copy_(x.cuda())
    assert xs.data_ptr() % 16 != 0
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    y = torch.empty((p.B, p.C_out) + O, dtype=p.torch_dtype, device="cuda")
    ct.ct_conv_transpose_nd(xs, w.cuda(), b.cuda(), y, None, p.stride, p.pad_lo, p.pad_hi,
                            p.dilation, p.output_padding, p.groups, ct.CT_ROUTE_TC_GEMM)
    torch.cuda.synchronize()
    assert_close(p, y, ref, "tc route, unaligned x")
