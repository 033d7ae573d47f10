"""GPU parity: the CUDA path against the fp64 oracle, element by element.

Every case draws seeded inputs from the shared generator, runs the library
through its C ABI (ctypes binding) and compares with oracle.conv_transpose
(full scatter) or oracle.points (sampled outputs), within the tolerance in
tests/_parity.py.  Each route is exercised on every problem it supports.
"""
import numpy as np
import pytest
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import (TOL, assert_close, check_full, max_err, run, sample_indices,
                     supported_routes)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transposed_convolution_convtranspose1_gb300 import _build
    _build.build_library()
    ct.lib()
    yield
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.CT_OK, f"device error word set after the module: {code:#x}"


# --------------------------------------------------------------------------
# the five named workloads, full size
# --------------------------------------------------------------------------

@pytest.mark.parametrize("i", range(5), ids=[p.name for p in synth.WORKLOADS])
def test_workload_full_oracle(i):
    p = synth.workload(i)
    err, scale = check_full(p)
    print(f"{p.name}: route {ct.ct_conv_transpose_route(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation, p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))} max|err| {err:.3e} max|y| {scale:.3e}")


@pytest.mark.parametrize("i", range(5), ids=[p.name for p in synth.WORKLOADS])
def test_workload_every_route_sampled(i):
    """Every route that supports the workload, checked on sampled outputs."""
    p = synth.workload(i)
    x, w, b = synth.make_inputs(p)
    rng = np.random.default_rng(100 + i)
    for r in supported_routes(p):
        y = run(p, x, w, b, route=r)
        torch.cuda.synchronize()
        yc = y.to(torch.float64).cpu().numpy()
        idx = sample_indices(yc.shape, 2000, rng)
        ref = oracle.points(x, w, b, idx, **p.attrs())
        got = yc[tuple(idx.T)]
        err = float(np.max(np.abs(got - ref)))
        scale = float(np.max(np.abs(ref)))
        assert err <= TOL[p.dtype] * max(scale, 1e-30), (p.name, r, err, scale)


# --------------------------------------------------------------------------
# seeded grid over nd, stride, pads, dilation, output_padding, groups, dtype
# --------------------------------------------------------------------------

def _grid(seed, n):
    r = np.random.default_rng(seed)
    probs = []
    for i in range(n):
        nd = int(r.integers(1, 4))
        dtype = ["f32", "bf16", "f16"][i % 3]
        g = int(r.choice([1, 1, 1, 2, 4]))
        Cig = int(r.choice([1, 3, 8, 16, 24, 64]))
        Cog = int(r.choice([1, 5, 8, 16, 40, 64]))
        if nd == 1:
            sp = (int(r.integers(1, 300)),)
        elif nd == 2:
            sp = (int(r.integers(1, 40)), int(r.integers(1, 70)))
        else:
            sp = (int(r.integers(1, 6)), int(r.integers(1, 14)), int(r.integers(1, 20)))
        k, s, d, pl, ph, op = [], [], [], [], [], []
        for a in range(nd):
            k.append(int(r.integers(1, 6)))
            s.append(int(r.integers(1, 4)))
            d.append(int(r.integers(1, 3)))
            op.append(int(r.integers(0, max(s[-1], d[-1]))))
            while True:
                lo, hi = int(r.integers(0, 4)), int(r.integers(0, 4))
                O = (sp[a] - 1) * s[-1] - lo - hi + d[-1] * (k[-1] - 1) + op[-1] + 1
                if O >= 1:
                    break
            pl.append(lo)
            ph.append(hi)
        B = int(r.integers(1, 4))
        probs.append(synth.problem(f"grid{seed}_{i}", B, g * Cig, g * Cog, sp, tuple(k),
                                   stride=tuple(s), pad_lo=tuple(pl), pad_hi=tuple(ph),
                                   dilation=tuple(d), output_padding=tuple(op), groups=g,
                                   bias=bool(r.random() < 0.75), dtype=dtype,
                                   seed=seed * 1000 + i))
    return probs


@pytest.mark.parametrize("p", _grid(1, 36), ids=lambda p: p.name)
def test_grid_every_route(p):
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    routes = supported_routes(p)
    assert ct.CT_ROUTE_GATHER in routes
    for r in [ct.CT_ROUTE_AUTO] + routes:
        y = run(p, x, w, b, route=r)
        torch.cuda.synchronize()
        assert_close(p, y, ref, f"route {r}")


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_empty_input_channels_gives_bias(dtype):
    p = synth.problem("cin0", 2, 0, 6, (5, 7), 3, stride=2, pad=1, dtype=dtype, seed=3)
    x, w, b = synth.make_inputs(p)
    assert ct.ct_conv_transpose_route(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo,
                                      p.pad_hi, p.dilation, p.output_padding, p.groups,
                                      ct.dtype_code(p.torch_dtype)) == ct.CT_ROUTE_BIAS_FILL
    y = run(p, x, w, b)
    torch.cuda.synchronize()
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    assert_close(p, y, ref)
    np.testing.assert_array_equal(
        y.float().cpu().numpy(),
        np.broadcast_to(b.float().numpy()[None, :, None, None], y.shape))


def test_zero_input_extent_with_nonempty_output():
    # I = 0 on one axis, but k and output_padding give O >= 1: only bias remains.
    p = synth.problem("i0", 1, 3, 4, (0, 5), (3, 2), stride=(2, 1), pad=(0, 0),
                      output_padding=(1, 0), dtype="f32", seed=4)
    x, w, b = synth.make_inputs(p)
    y = run(p, x, w, b)
    torch.cuda.synchronize()
    assert y.shape == (1, 4, (0 - 1) * 2 + 2 + 1 + 1, 6)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    assert_close(p, y, ref)


def test_zero_batch_launches_nothing():
    p = synth.problem("b0", 0, 4, 4, (6,), 3, stride=2, dtype="f32", seed=5)
    x, w, b = synth.make_inputs(p)
    y = run(p, x, w, b)
    torch.cuda.synchronize()
    assert y.shape == (0, 4, 13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_phases_without_taps(dtype):
    # stride 5 > k*d: 2 of 5 residues per axis get taps, the rest only bias
    p = synth.problem("sparse_phase", 2, 16, 16, (9, 11), 2, stride=5, pad=0,
                      output_padding=(4, 3), dtype=dtype, seed=6)
    for r in supported_routes(p):
        check_full(p, route=r)


def test_no_bias_and_1x1_stride1():
    p = synth.problem("1x1", 3, 32, 24, (17, 19), 1, dtype="f32", bias=False, seed=9)
    check_full(p)
    p = p.replace(dtype="bf16", name="1x1bf16")
    check_full(p)


def test_dilation_larger_than_stride_with_output_padding():
    p = synth.problem("d3s1op2", 2, 8, 8, (13,), 3, stride=1, dilation=3, pad_lo=2, pad_hi=4,
                      output_padding=2, dtype="f32", seed=10)
    for r in supported_routes(p):
        check_full(p, route=r)


# --------------------------------------------------------------------------
# determinism, guard bands, streams, host entry point
# --------------------------------------------------------------------------

@pytest.mark.parametrize("i", [1, 2, 3, 4])
def test_deterministic_bits(i):
    p = synth.workload(i)
    x, w, b = synth.make_inputs(p)
    y1 = run(p, x, w, b)
    y2 = run(p, x, w, b)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16) if y1.element_size() == 2 else y1.view(torch.int32),
                       y2.view(torch.int16) if y2.element_size() == 2 else y2.view(torch.int32))


@pytest.mark.parametrize("p", [synth.workload(0),
                               synth.problem("guard_bf16", 2, 64, 48, (10, 13), 4, stride=2,
                                             pad=1, dtype="bf16", seed=11),
                               synth.problem("guard_1d", 3, 40, 24, (77,), 8, stride=4, pad=2,
                                             dtype="f32", seed=12)],
                         ids=lambda p: p.name)
def test_guard_bands_survive(p):
    """y sits inside a larger buffer whose margins hold a sentinel pattern."""
    x, w, b = synth.make_inputs(p)
    xd, wd, bd = x.cuda(), w.cuda(), (None if b is None else b.cuda())
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    n = p.B * p.C_out * int(np.prod(O))
    margin = 4096
    buf = torch.full((n + 2 * margin,), -12345.0, dtype=p.torch_dtype, device="cuda")
    y = buf[margin:margin + n].view((p.B, p.C_out) + O)
    for r in supported_routes(p):
        ct.ct_conv_transpose_nd(xd, wd, bd, y, None, p.stride, p.pad_lo, p.pad_hi, p.dilation,
                                p.output_padding, p.groups, r)
        torch.cuda.synchronize()
        sentinel = torch.tensor(-12345.0, dtype=p.torch_dtype).item()
        assert bool((buf[:margin] == sentinel).all()) and bool((buf[margin + n:] == sentinel).all()), r
        ref = oracle.conv_transpose(x, w, b, **p.attrs())
        assert_close(p, y, ref, f"route {r}")


def test_side_stream_and_explicit_workspace():
    p = synth.workload(2)
    x, w, b = synth.make_inputs(p)
    nbytes = ct.ct_conv_transpose_workspace_bytes(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride,
                                                  p.pad_lo, p.pad_hi, p.dilation,
                                                  p.output_padding, p.groups,
                                                  ct.dtype_code(p.torch_dtype))
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda") if nbytes else None
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = run(p, x, w, b, workspace=ws, stream=s)
    s.synchronize()
    y0 = run(p, x, w, b)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    if nbytes:
        small = torch.empty(nbytes - 256, dtype=torch.uint8, device="cuda")
        with pytest.raises(ct.CtError) as e:
            run(p, x, w, b, workspace=small)
        assert e.value.status == ct.ct.CT_ERR_WORKSPACE


@pytest.mark.parametrize("i", [0, 1, 2, 3])
def test_host_entry_point_matches_device(i):
    p = synth.workload(i)
    x, w, b = synth.make_inputs(p)
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    yh = torch.empty((p.B, p.C_out) + O, dtype=p.torch_dtype).pin_memory()
    ct.ct_conv_transpose_nd_host(x.pin_memory(), w.pin_memory(),
                                 None if b is None else b.pin_memory(), yh, p.stride, p.pad_lo,
                                 p.pad_hi, p.dilation, p.output_padding, p.groups)
    yd = run(p, x, w, b)
    torch.cuda.synchronize()
    assert torch.equal(yh, yd.cpu())


def test_host_entry_point_pipeline_chunks_stream_and_release():
    """B = 11 runs as 6 batch chunks of 2 (the last of 1) through the copy /
    compute / copy pipeline; the result equals the device call's bit for bit,
    on the default stream and on a caller's stream, before and after the
    library's pool memory is released."""
    p = synth.problem("host_chunks", 11, 48, 40, (3000,), 8, stride=4, pad=2, seed=901)
    x, w, b = synth.make_inputs(p)
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    hx, hw, hb = x.pin_memory(), w.pin_memory(), b.pin_memory()
    yd = run(p, x, w, b)
    torch.cuda.synchronize()
    ref = yd.cpu()
    s = torch.cuda.Stream()
    for stream in (None, s, None):
        yh = torch.full((p.B, p.C_out) + O, float("nan"), dtype=p.torch_dtype).pin_memory()
        ct.ct_conv_transpose_nd_host(hx, hw, hb, yh, p.stride, p.pad_lo, p.pad_hi, p.dilation,
                                     p.output_padding, p.groups, stream=stream)
        assert torch.equal(yh, ref)
        ct.ct_host_buffers_release()

