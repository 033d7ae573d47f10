"""GPU parity of the backward pass (dx, dw, db) against the fp64 oracle.

The oracle's gradients are the adjoint of its scatter-add, pinned in
test_oracle_backward_pins.  Bars: max|g - g_oracle| <= 1e-5 * max|g_oracle|
for fp32 and 1e-2 * max|g_oracle| for bf16/fp16 (each gradient on its own),
computed on the values the device sees (16-bit inputs widened exactly).
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
    yield


def _dy_for(p, seed):
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    g = torch.Generator().manual_seed(seed)
    return torch.randn((p.B, p.C_out) + tuple(O), generator=g).to(p.torch_dtype)


def _gpu_grads(p, x, w, dy, need=("dx", "dw", "db")):
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    dx = torch.full_like(xd, float("nan")) if "dx" in need else None
    dw = torch.full_like(wd, float("nan")) if "dw" in need else None
    db = torch.full((p.C_out,), float("nan"), dtype=dyd.dtype, device="cuda") if "db" in need else None
    ct.ct_conv_transpose_backward_nd(xd, wd, dyd, dx, dw, db, None, p.stride, p.pad_lo, p.pad_hi,
                                     p.dilation, p.output_padding, p.groups)
    torch.cuda.synchronize()
    return dx, dw, db


def _check(p, got, ref, what):
    if ref.size == 0:
        assert got.numel() == 0
        return
    g = got.to(torch.float64).cpu().numpy()
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(g - ref)))
    assert np.isfinite(g).all(), f"{p.name} {what}: non-finite values"
    assert err <= TOL[p.dtype] * scale + 1e-30, f"{p.name} {what}: max|err| {err:.3e} > {TOL[p.dtype]:.0e} * {scale:.3e}"


def _check_all(p, seed=0):
    x, w, _ = synth.make_inputs(p)
    dy = _dy_for(p, 1000 + seed)
    rdx, rdw, rdb = oracle.conv_transpose_backward(x, w, dy, **p.attrs())
    dx, dw, db = _gpu_grads(p, x, w, dy)
    _check(p, dx, rdx, "dx")
    _check(p, dw, rdw, "dw")
    _check(p, db, rdb, "db")


def _grid():
    r = np.random.default_rng(1234)
    out = []
    for n in range(30):
        nd = int(r.integers(1, 4))
        G = int(r.choice([1, 1, 2, 4]))
        Cig, Cog = int(r.integers(1, 20)), int(r.integers(1, 20))
        spatial, k, s, pl, ph, d, op = [], [], [], [], [], [], []
        for _ in range(nd):
            spatial.append(int(r.integers(1, 12 if nd < 3 else 6)))
            k.append(int(r.integers(1, 5)))
            s.append(int(r.integers(1, 4)))
            d.append(int(r.integers(1, 3)))
            op.append(int(r.integers(0, max(s[-1], d[-1]))))
            while True:
                a, b = int(r.integers(0, 3)), int(r.integers(0, 3))
                if (spatial[-1] - 1) * s[-1] - a - b + d[-1] * (k[-1] - 1) + op[-1] + 1 >= 1:
                    break
            pl.append(a)
            ph.append(b)
        dtype = str(r.choice(["f32", "f32", "bf16", "f16"]))
        out.append(P(f"bwd{n}_{nd}d_{dtype}_g{G}", int(r.integers(1, 4)), G * Cig, G * Cog,
                     tuple(spatial), tuple(k), stride=tuple(s), pad_lo=tuple(pl), pad_hi=tuple(ph),
                     dilation=tuple(d), output_padding=tuple(op), groups=G, dtype=dtype,
                     seed=2000 + n))
    return out


@pytest.mark.parametrize("p", _grid(), ids=lambda p: p.name)
def test_backward_grid_matches_oracle(p):
    _check_all(p)


# Small channel groups (at most 8 input and 8 output channels each), the
# shapes of the dedicated grouped dw kernel: 1-D, 2-D and 3-D, dilation, ragged
# bands (H not a multiple of 4), 25 taps, a 1x1 kernel, and one with 36 taps
# (beyond that kernel, so the general dw kernel takes it).
SMALL_GROUPS = [
    P("sg_2d_full8", 2, 64, 64, (13, 10), 3, stride=2, pad=1, dilation=2, output_padding=1,
      groups=8, seed=3001),
    P("sg_2d_5x7_k5", 1, 15, 21, (9, 11), 5, stride=(1, 2), pad=2, groups=3, seed=3002),
    P("sg_3d", 2, 16, 12, (3, 6, 5), 3, stride=(2, 1, 2), pad=1, output_padding=(1, 0, 1),
      groups=2, seed=3003),
    P("sg_1d", 3, 12, 16, (37,), 4, stride=3, pad=1, dilation=2, groups=4, seed=3004),
    P("sg_k1", 2, 8, 8, (7, 7), 1, stride=2, groups=2, seed=3005),
    P("sg_36taps", 1, 8, 8, (4, 5, 6), (3, 3, 4), stride=2, pad=1, groups=2, seed=3006),
    P("sg_bf16", 2, 32, 32, (10, 12), 4, stride=2, pad=1, groups=4, dtype="bf16", seed=3007),
    P("sg_f16_c1", 2, 6, 6, (5, 9), 3, stride=2, groups=6, dtype="f16", seed=3008),
    # fp32 (staged by bulk row copies): widths that are not multiples of 4,
    # a 3-D kernel, pad_lo 6 on W, many bands
    P("sg_tma_2d", 2, 32, 24, (13, 16), 3, stride=2, pad=1, output_padding=1, groups=4, seed=3009),
    P("sg_tma_3d", 1, 16, 16, (3, 6, 8), 3, stride=(2, 1, 2), pad=1, output_padding=(1, 0, 1),
      groups=2, seed=3010),
    P("sg_tma_k5_pad6", 1, 10, 14, (9, 12), 5, stride=(1, 2), pad=(2, 6), output_padding=(0, 1),
      groups=2, seed=3011),
    P("sg_tma_many_bands", 3, 8, 8, (41, 8), (2, 4), stride=(1, 4), pad=(0, 0), groups=1,
      seed=3012),
]


@pytest.mark.parametrize("p", SMALL_GROUPS, ids=lambda p: p.name)
def test_backward_small_groups_match_oracle(p):
    _check_all(p, seed=3)


# 16-bit types, groups of 1, at least 16 channels each side: dx on the tcgen05
# GEMM (dy's channels-last copy read by TMA boxes with element strides equal
# to the stride).  Channel counts off the 64/128 tiles, odd extents, strides 1
# to 4 (W stride 4: boxes 64 positions wide), 1-D and 3-D, dilation,
# asymmetric pads, output_padding, 8 taps on an axis, a row wider than a tile.
TC_DX = [
    P("tcdx_2d_bf16", 2, 32, 48, (9, 12), 4, stride=2, pad=1, dtype="bf16", seed=3101),
    P("tcdx_3d_f16", 1, 24, 40, (3, 6, 10), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
      dtype="f16", seed=3102),
    P("tcdx_1d_dil", 3, 64, 16, (37,), 5, stride=3, pad_lo=(2,), pad_hi=(4,), dilation=2,
      dtype="bf16", seed=3103),
    P("tcdx_k8_s4", 1, 16, 130, (5, 7), 8, stride=4, pad=2, dtype="bf16", seed=3104),
    P("tcdx_wide", 1, 80, 24, (3, 200), 3, stride=(1, 2), pad=1, output_padding=(0, 1), dtype="bf16",
      seed=3105),
    P("tcdx_s1", 2, 40, 72, (6, 7, 5), (2, 3, 2), stride=1, pad=(1, 0, 1), dtype="f16", seed=3106),
]


def test_backward_kernel_query_names_the_kernels_that_run():
    """The query's answers on the workloads and on the shapes of each dx/dw
    kernel class (the tensor-core dx on 16-bit problems of one group, the
    small-group dw on groups of at most 8 channels)."""
    def names(p):
        return ct.ct_conv_transpose_backward_kernels(
            p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
            p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))
    assert names(synth.workload(2)) == ("tc_phase_gemm", "tc_dw_gemm")
    assert names(synth.workload(4)) == ("tc_phase_gemm", "tc_dw_gemm")
    assert names(synth.workload(1)) == ("tc32_phase_gemm", "bwd_dw_kernel")
    assert names(synth.workload(3)) == ("bwd_dx_kernel", "bwd_dw_grouped_kernel")
    for p in TC_DX:
        assert names(p)[0] == "tc_phase_gemm", p.name
    for p in TC_DW:
        assert names(p)[1] == "tc_dw_gemm", p.name
    for p in TC32_DX:
        assert names(p)[0] == "tc32_phase_gemm", p.name
    for p in SMALL_GROUPS:
        if p.name != "sg_36taps":
            assert names(p)[1] == "bwd_dw_grouped_kernel", p.name


# dw on the tcgen05 GEMM (16-bit, one group, >= 16 channels, W stride <= 4,
# input width a multiple of 8): x K-major from its own layout, dy MN-major from
# its channels-last copy read with element strides; several input- and
# output-channel blocks and tap pairs (an odd tap count), rows longer than a
# 64-position block, 1-D and 3-D, dilation, asymmetric pads, W stride 4.
TC_DW = [
    P("tcdw_2d", 2, 32, 48, (9, 16), 4, stride=2, pad=1, dtype="bf16", seed=3201),
    P("tcdw_3d_f16", 1, 24, 40, (3, 6, 16), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
      dtype="f16", seed=3202),
    P("tcdw_1d_dil", 3, 64, 16, (40,), 5, stride=3, pad_lo=(2,), pad_hi=(4,), dilation=2,
      dtype="bf16", seed=3203),
    P("tcdw_wide", 1, 80, 24, (3, 200), 3, stride=(1, 2), pad=1, output_padding=(0, 1), dtype="bf16",
      seed=3204),
    P("tcdw_blocks", 1, 160, 136, (4, 8), 2, stride=2, dtype="bf16", seed=3205),
    P("tcdw_s4", 1, 16, 130, (5, 8), 8, stride=4, pad=2, dtype="bf16", seed=3206),
]


@pytest.mark.parametrize("p", TC_DW, ids=lambda p: p.name)
def test_backward_tensor_core_dw_matches_oracle(p):
    x, w, _ = synth.make_inputs(p)
    dy = _dy_for(p, 78)
    _, rdw, _ = oracle.conv_transpose_backward(x, w, dy, **p.attrs(), need=("dw",))
    _, dw, _ = _gpu_grads(p, x, w, dy, need=("dw",))
    _check(p, dw, rdw, "dw")


# fp32 dx on the error-compensated TF32 GEMM (one group, >= 32 channels): the
# same mapping; a 1-D row of 300 positions at stride 4 takes four boxes per
# tile row, and a 2-D and a 3-D case with dilation and output_padding.
TC32_DX = [
    P("tc32dx_1d_s4", 2, 64, 48, (300,), 8, stride=4, pad=2, seed=3301),
    P("tc32dx_2d", 2, 40, 72, (9, 12), 3, stride=2, pad=1, output_padding=1, seed=3302),
    P("tc32dx_3d_dil", 1, 32, 33, (3, 5, 8), 3, stride=(1, 2, 2), pad=1, dilation=(1, 2, 1),
      output_padding=(0, 1, 1), seed=3303),
]


@pytest.mark.parametrize("p", TC32_DX, ids=lambda p: p.name)
def test_backward_tf32_dx_matches_oracle(p):
    x, w, _ = synth.make_inputs(p)
    dy = _dy_for(p, 79)
    rdx, _, _ = oracle.conv_transpose_backward(x, w, dy, **p.attrs(), need=("dx",))
    dx, _, _ = _gpu_grads(p, x, w, dy, need=("dx",))
    _check(p, dx, rdx, "dx")


@pytest.mark.parametrize("p", TC_DX, ids=lambda p: p.name)
def test_backward_tensor_core_dx_matches_oracle(p):
    x, w, _ = synth.make_inputs(p)
    dy = _dy_for(p, 77)
    rdx, _, _ = oracle.conv_transpose_backward(x, w, dy, **p.attrs(), need=("dx",))
    dx, _, _ = _gpu_grads(p, x, w, dy, need=("dx",))
    _check(p, dx, rdx, "dx")


def test_grouped_dw_does_not_depend_on_pointer_alignment():
    """The small-group dw kernel stages fp32 rows by bulk copies widened to
    16-byte boundaries, so x and dy may start anywhere a float may: views one
    and three floats into their buffers must give the same dw, bit for bit,
    as 256-byte aligned tensors (the same products summed in the same order)."""
    p = P("sg_align", 2, 32, 32, (14, 20), 3, stride=2, pad=2, dilation=2, output_padding=1,
          groups=4, seed=3013)
    x, w, _ = synth.make_inputs(p)
    dy = _dy_for(p, 77)
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()

    def shifted(t, k):
        buf = torch.empty(t.numel() + k, device="cuda")
        v = buf[k:].view_as(t)
        v.copy_(t)
        return v

    x1, dy3 = shifted(xd, 1), shifted(dyd, 3)
    assert x1.data_ptr() % 16 != 0 and dy3.data_ptr() % 16 != 0
    out = []
    for xi, dyi in ((xd, dyd), (x1, dy3)):
        dw = torch.full_like(wd, float("nan"))
        ct.ct_conv_transpose_backward_nd(xi, wd, dyi, None, dw, None, None, p.stride, p.pad_lo,
                                         p.pad_hi, p.dilation, p.output_padding, p.groups)
        out.append(dw)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])
    _, rdw, _ = oracle.conv_transpose_backward(x, w, dy, **p.attrs(), need=("dw",))
    _check(p, out[0], rdw, "dw")


@pytest.mark.parametrize("i", [0, 1, 3])
def test_backward_workload_matches_oracle(i):
    _check_all(synth.workload(i))


def test_backward_bf16_workload_matches_oracle():
    p = synth.workload(2).replace(B=2)  # the 2-D bf16 workload, batch 2
    _check_all(p)


def test_backward_is_bit_reproducible_and_partial_requests_agree():
    p = synth.workload(3).replace(B=2)
    x, w, _ = synth.make_inputs(p)
    dy = _dy_for(p, 5)
    a = _gpu_grads(p, x, w, dy)
    b = _gpu_grads(p, x, w, dy)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    only_dw = _gpu_grads(p, x, w, dy, need=("dw",))
    assert only_dw[0] is None and only_dw[2] is None
    assert torch.equal(only_dw[1], a[1])
    only_dx = _gpu_grads(p, x, w, dy, need=("dx",))
    assert torch.equal(only_dx[0], a[0])


def test_backward_empty_batch_gives_zero_weight_and_bias_gradients():
    p = P("bwd_empty", 0, 4, 6, (5,), 3, stride=2)
    x = torch.zeros((0, 4, 5))
    w = synth.make_inputs(p.replace(B=1))[1]
    dy = torch.zeros((0, 6, 11))
    dx, dw, db = _gpu_grads(p, x, w, dy)
    assert dx.numel() == 0
    assert torch.equal(dw.cpu(), torch.zeros_like(w))
    assert torch.equal(db.cpu(), torch.zeros(6))


def test_autograd_function_matches_torch():
    """ConvTransposeFunction's fp32 gradients against torch's own
    conv_transpose2d autograd run in float64 on the same values, within the
    fp32 bound relative to the largest gradient."""
    p = P("autograd", 2, 16, 24, (9, 7), 3, stride=2, pad=1, output_padding=1, seed=77)
    x, w, b = synth.make_inputs(p)
    dy = _dy_for(p, 9)
    x0, w0, b0 = (t.cuda().requires_grad_(True) for t in (x, w, b))
    x1, w1, b1 = (t.cuda().double().requires_grad_(True) for t in (x, w, b))
    y0 = ct.conv_transpose_autograd(x0, w0, b0, stride=2, padding=1, output_padding=1)
    y1 = torch.nn.functional.conv_transpose2d(x1, w1, b1, stride=2, padding=1, output_padding=1)
    assert float((y0.double() - y1).detach().abs().max()) <= 1e-5 * float(y1.detach().abs().max())
    y0.backward(dy.cuda())
    y1.backward(dy.cuda().double())
    for a, c in ((x0.grad, x1.grad), (w0.grad, w1.grad), (b0.grad, b1.grad)):
        scale = float(c.abs().max())
        assert float((a.double() - c).abs().max()) <= 1e-5 * scale
