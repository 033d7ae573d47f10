"""GPU parity of the grouped route on groups of 5..8 input and output
channels (2-D/3-D outputs) against the fp64 oracle, with guard bands around y.

The problems cover: the grouped workload's geometry (one live W residue:
2-wide stores, bias-only rows and columns), both W residues live, W strides
1 and 3, odd output widths, input rows wider than the staged kernel's span
(direct kernel), ragged bands along H, mixed strides with dilation and
asymmetric pads, a 3-D output with a D stride, no bias, 16-bit dtypes, and
an output that is only 4-byte aligned (2-wide stores off).  The fp32 problems
whose input width is a multiple of 4 take one of the two kernels whose input
rows arrive by TMA boxes (channel boxes past the last channel, rows and
columns outside the input read as zero): the warp-pair kernel where four
pairs' buffers fit in shared memory, the TMA block kernel otherwise (3-D
problems with three or four D taps); each problem names the kernel it must
take.
The warp-pair problems add several W chunks per row, ragged bands of 3
rows, output depths no tap reaches, an H offset span of 3, a fused activation
and more items than warps.
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


SHAPES = [
    P("g_workload_geom", 1, 16, 16, (56, 56), 3, stride=2, pad=1, dilation=2, output_padding=1,
      groups=2, seed=701),
    P("g_k4s2", 2, 8, 8, (20, 30), 4, stride=2, pad=1, seed=702),
    P("g_cig5_cog7_nobias", 2, 5, 7, (13, 70), 3, stride=2, pad=1, output_padding=1, seed=703,
      bias=False),
    P("g_s13_d12", 1, 12, 12, (17, 9), (3, 5), stride=(1, 3), pad_lo=(0, 2), pad_hi=(1, 1),
      dilation=(1, 2), output_padding=(0, 2), groups=2, seed=704),
    P("g_s34", 1, 8, 5, (9, 40), (5, 3), stride=(3, 4), pad_lo=(2, 0), pad_hi=(0, 1),
      output_padding=(2, 3), seed=705),
    P("g_3d", 1, 16, 16, (3, 12, 10), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
      groups=2, seed=706),
    P("g_wide_s1", 1, 7, 8, (30, 130), 3, stride=1, pad=1, seed=707),
    P("g_bf16", 2, 32, 32, (24, 40), 3, stride=2, pad=1, dilation=2, output_padding=1, groups=4,
      dtype="bf16", seed=708),
    P("g_f16_k4", 1, 24, 24, (18, 22), 4, stride=2, pad=1, groups=3, dtype="f16", seed=709),
    P("g_ragged_h", 3, 6, 6, (37, 33), 3, stride=2, pad=1, output_padding=1, seed=710),
    # fp32 with input widths a multiple of 4: input rows staged by TMA boxes
    P("g_tma_cig5_cog7", 2, 15, 21, (20, 72), 3, stride=2, pad=1, output_padding=1, groups=3,
      seed=711, bias=False),
    P("g_tma_k4s2", 1, 8, 8, (20, 32), 4, stride=2, pad=1, seed=712),
    P("g_tma_s13", 1, 12, 12, (17, 12), 3, stride=(1, 3), pad_lo=(0, 2), pad_hi=(1, 1),
      dilation=(1, 2), output_padding=(0, 2), groups=2, seed=713),
    P("g_tma_3d", 1, 16, 16, (3, 12, 12), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
      groups=2, seed=714),
    P("g_tma_wide_s1", 1, 7, 8, (30, 132), 3, stride=1, pad=1, seed=715),
    P("g_tma_ragged", 3, 6, 6, (37, 36), 3, stride=2, pad=1, output_padding=1, seed=716),
    # warp-pipeline kernel: D stride 2 with a D residue no tap reaches, H span 3
    P("g_warp_3d_dead_d", 2, 16, 16, (3, 10, 16), (1, 3, 3), stride=2, pad=(0, 1, 1),
      output_padding=(1, 1, 1), groups=2, seed=717),
    P("g_warp_span3", 1, 8, 8, (14, 24), (4, 3), stride=(1, 2), pad_lo=(3, 1), pad_hi=(0, 1),
      dilation=(1, 2), output_padding=(0, 1), seed=718),
    P("g_warp_many_items", 8, 128, 128, (40, 44), 3, stride=2, pad=1, dilation=2,
      output_padding=1, groups=16, seed=719),
    # four D taps: too much shared memory for the warp pairs: the TMA block kernel
    P("g_tma_3d_k4", 1, 16, 16, (5, 12, 12), (4, 3, 3), stride=(1, 2, 2), pad=1,
      output_padding=(0, 1, 1), groups=2, seed=720),
]

# the kernel each fp32 TMA-eligible problem must take
KERNEL = {"g_workload_geom": "grouped_warp_kernel", "g_tma_cig5_cog7": "grouped_warp_kernel",
          "g_tma_k4s2": "grouped_warp_kernel", "g_tma_s13": "grouped_warp_kernel",
          "g_tma_3d": "grouped_tma_kernel", "g_tma_3d_k4": "grouped_tma_kernel", "g_tma_wide_s1": "grouped_warp_kernel",
          "g_tma_ragged": "grouped_warp_kernel", "g_warp_3d_dead_d": "grouped_warp_kernel",
          "g_warp_span3": "grouped_warp_kernel", "g_warp_many_items": "grouped_warp_kernel"}


def _kernel(p):
    return ct.ct_conv_transpose_kernel(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo,
                                       p.pad_hi, p.dilation, p.output_padding, p.groups,
                                       ct.dtype_code(p.torch_dtype))


def _check(p, pad_elems=64):
    if p.name in KERNEL:
        assert _kernel(p) == KERNEL[p.name], (p.name, _kernel(p))
    x, w, b = synth.make_inputs(p)
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
                                       p.output_padding)
    shape = (p.B, p.C_out) + tuple(O)
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad_elems,), float("nan"), dtype=p.torch_dtype, device="cuda")
    y = buf[pad_elems:pad_elems + n].view(shape)
    ct.ct_conv_transpose_nd(x.cuda(), w.cuda(), None if b is None else b.cuda(), y, None,
                            p.stride, p.pad_lo, p.pad_hi, p.dilation, p.output_padding, p.groups,
                            ct.CT_ROUTE_GROUPED)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:pad_elems].float()).all() and torch.isnan(buf[pad_elems + n:].float()).all()
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    got = y.to(torch.float64).cpu().numpy()
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - ref)))
    scale = float(np.max(np.abs(ref)))
    assert err <= TOL[p.dtype] * scale, f"{p.name}: {err:.3e} > {TOL[p.dtype]} * {scale:.3e}"


@pytest.mark.parametrize("p", SHAPES, ids=lambda p: p.name)
def test_grouped_route_matches_oracle(p):
    _check(p)


def test_grouped_route_with_a_4_byte_aligned_output():
    """y one fp32 element past an 8-byte boundary: the 2-wide stores must be
    off, the scalar ones give the same result."""
    _check(SHAPES[0], pad_elems=1)


def test_grouped_route_is_deterministic():
    p = SHAPES[1]
    x, w, b = synth.make_inputs(p)
    outs = []
    for _ in range(2):
        O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                           p.dilation, p.output_padding)
        y = torch.empty((p.B, p.C_out) + tuple(O), device="cuda")
        ct.ct_conv_transpose_nd(x.cuda(), w.cuda(), b.cuda(), y, None, p.stride, p.pad_lo,
                                p.pad_hi, p.dilation, p.output_padding, p.groups,
                                ct.CT_ROUTE_GROUPED)
        outs.append(y)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("act", ["relu", "gelu", "sigmoid"])
def test_grouped_warp_kernel_fuses_the_activation(act):
    """The warp-pair kernel applies the activation in its epilogue (to
    computed outputs and to the bias-only ones): y = act(convT(x) + b)."""
    p = SHAPES[0]
    assert _kernel(p) == "grouped_warp_kernel"
    x, w, b = synth.make_inputs(p)
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
                                       p.output_padding)
    y = torch.full((p.B, p.C_out) + tuple(O), float("nan"), device="cuda")
    ct.ct_conv_transpose_nd_ex(x.cuda(), w.cuda(), b.cuda(), y, None, p.stride, p.pad_lo,
                               p.pad_hi, p.dilation, p.output_padding, p.groups,
                               activation=act)
    torch.cuda.synchronize()
    ref = oracle.activation(oracle.conv_transpose(x, w, b, **p.attrs()), act)
    got = y.double().cpu().numpy()
    err = float(np.max(np.abs(got - ref)))
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    assert err <= TOL[p.dtype] * scale, f"{act}: {err:.3e} > {TOL[p.dtype]} * {scale:.3e}"
