"""GPU parity of the fp32 tcgen05 route (error-compensated TF32: every fp32
operand split into TF32 hi + lo parts, products accumulated as
hi*hi + hi*lo + lo*hi in fp32).

The bar is the fp32 one, max|y - y_oracle| <= 1e-5 * max|y_oracle|, and a
tighter check on a deep reduction shows the route is far more accurate than
a single TF32 product (10-bit mantissa) would allow.  Shapes hit the route's
corners: one stride phase per tile with 256 positions laid out as 1..8 rows
of 256..32 W positions, ragged tails on every axis, C_in not a multiple of
the 32-channel k-block, C_out not a multiple of 128, strides 1..8, phases
without taps (bias only), 1-D/2-D/3-D, dilation, asymmetric pads and
output_padding.
"""
import numpy as np
import pytest
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import assert_close, max_err, run, supported_routes

pytestmark = pytest.mark.gpu

P = synth.problem
CASES = [
    P("tc32_1d_c1_like", 2, 96, 72, (300,), 8, stride=4, pad=2, seed=501),
    P("tc32_1d_s1", 2, 40, 130, (257,), 5, stride=1, pad=2, seed=502),
    P("tc32_1d_s3_dil", 1, 33, 48, (101,), 4, stride=3, pad_lo=1, pad_hi=3, dilation=2,
      output_padding=2, seed=503),
    P("tc32_1d_s8", 1, 64, 64, (64,), 16, stride=8, pad=4, seed=504),
    P("tc32_1d_long", 1, 64, 40, (1100,), 4, stride=2, pad=1, seed=505),
    P("tc32_2d_rows", 2, 64, 40, (13, 21), 4, stride=2, pad=1, seed=506),
    P("tc32_2d_wide", 1, 32, 32, (5, 600), (3, 2), stride=(1, 2), pad=(1, 0), seed=507),
    P("tc32_2d_empty_phases", 1, 32, 32, (6, 7), 2, stride=5, output_padding=(4, 3), seed=508),
    P("tc32_2d_dilated", 2, 48, 64, (12, 12), 3, stride=2, pad=1, dilation=2,
      output_padding=1, seed=509),
    P("tc32_3d", 1, 32, 48, (3, 7, 9), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
      seed=510),
    P("tc32_3d_s2", 1, 32, 32, (4, 5, 6), (2, 3, 3), stride=2, pad=(0, 1, 1), seed=511),
    P("tc32_no_bias", 3, 48, 64, (77,), 3, stride=2, pad=1, bias=False, seed=512),
    P("tc32_two_oc_tiles", 1, 64, 260, (9, 9), 4, stride=2, pad=1, seed=513),
    P("tc32_big_k", 1, 512, 64, (8, 8), 4, stride=2, pad=1, seed=514),
    P("tc32_1x1", 2, 128, 96, (33, 31), 1, seed=515),
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
def test_tc32_route_matches_oracle(p):
    assert ct.CT_ROUTE_TC32_GEMM in supported_routes(p), p.name
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    y = run(p, x, w, b, route=ct.CT_ROUTE_TC32_GEMM)
    torch.cuda.synchronize()
    assert_close(p, y, ref, "tc32 route")
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.CT_OK, f"{p.name}: device error word {code:#x}"


def test_tc32_accuracy_on_a_deep_reduction():
    """K = 1024 products per output (512 channels x 2 taps).  Plain TF32
    products (2^-11 relative rounding of each operand) would leave errors of
    order 1e-4 of max|y| at this depth; the hi/lo split must stay within
    2e-6 of max|y|, a fifth of the fp32 tolerance."""
    p = P("tc32_deep", 1, 512, 128, (256,), 8, stride=4, pad=2, seed=516)
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    y = run(p, x, w, b, route=ct.CT_ROUTE_TC32_GEMM)
    torch.cuda.synchronize()
    err, scale = max_err(y, ref)
    assert err <= 2e-6 * scale, (err, scale)


def test_tc32_matches_simt_route():
    """The tensor-core and the CUDA-core fp32 routes agree within the sum of
    their fp32 error bounds on the same inputs."""
    p = P("tc32_vs_simt", 2, 128, 96, (200,), 8, stride=4, pad=2, seed=517)
    x, w, b = synth.make_inputs(p)
    yt = run(p, x, w, b, route=ct.CT_ROUTE_TC32_GEMM)
    ys = run(p, x, w, b, route=ct.CT_ROUTE_SIMT_GEMM)
    torch.cuda.synchronize()
    scale = float(ys.abs().max())
    assert float((yt - ys).abs().max()) <= 2e-5 * scale


def test_auto_route_is_tc32_for_dense_fp32():
    p = synth.workload(1)
    r = ct.ct_conv_transpose_route(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo,
                                   p.pad_hi, p.dilation, p.output_padding, p.groups,
                                   ct.dtype_code(p.torch_dtype))
    assert r == ct.CT_ROUTE_TC32_GEMM


def test_tc32_route_rejects_grouped_and_16_bit():
    p = synth.problem("g2", 1, 64, 64, (8, 8), 3, stride=2, groups=2)
    assert ct.CT_ROUTE_TC32_GEMM not in supported_routes(p)
    p = synth.problem("bf16", 1, 64, 64, (8, 8), 3, stride=2, dtype="bf16")
    assert ct.CT_ROUTE_TC32_GEMM not in supported_routes(p)


def test_tc32_route_with_unaligned_x():
    """x starting 4 bytes past a 16-byte boundary: the layout pass reads it
    element by element, so results must not change."""
    p = P("tc32_unaligned", 2, 64, 32, (7, 9), 3, stride=2, pad=1, seed=518)
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    flat = torch.empty(x.numel() + 4, dtype=x.dtype, device="cuda")
    xs = flat[1:1 + x.numel()].view(x.shape)
    xs.copy_(x.cuda())
    assert xs.data_ptr() % 16 != 0
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    y = torch.empty((p.B, p.C_out) + O, dtype=p.torch_dtype, device="cuda")
    ct.ct_conv_transpose_nd(xs, w.cuda(), b.cuda(), y, None, p.stride, p.pad_lo, p.pad_hi,
                            p.dilation, p.output_padding, p.groups, ct.CT_ROUTE_TC32_GEMM)
    torch.cuda.synchronize()
    assert_close(p, y, ref, "tc32 route, unaligned x")


def test_tc32_full_size_sampled():
    """The 1-D fp32 workload (8 x 512 -> 256, L 2048, k 8, s 4) at full size,
    in the launch configuration the benchmark times, against the oracle at
    sampled outputs (and every corner)."""
    p = synth.workload(1)
    x, w, b = synth.make_inputs(p)
    y = run(p, x, w, b, route=ct.CT_ROUTE_TC32_GEMM)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    idx = np.stack([rng.integers(0, s, size=3000) for s in y.shape], axis=1)
    want = oracle.points(x, w, b, idx, **p.attrs())
    got = y.double().cpu().numpy()[tuple(idx.T)]
    scale = float(y.abs().max())
    assert float(np.max(np.abs(got - want))) <= 1e-5 * scale
