"""GPU parity at the library's size limits.

- The largest kernel and stride per axis the planner accepts (32), on every
  route that takes them, against the full fp64 oracle.
- Outputs with more than 2^31 elements, so that every flat index into y (and
  into the channels-last workspace) must be 64-bit: 1-D problems with a large
  stride (output 8x or 4x the input) through the TF32, bf16, grouped and
  generic routes, checked at sampled outputs (including the last ones and
  those around flat index 2^31) that the oracle evaluates one by one.  Each
  case holds up to about 10 GB on the device.
"""
import numpy as np
import pytest
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import TOL, assert_close, run, supported_routes

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


MAX_KS = [
    P("k32_s32_1d", 2, 3, 5, (7,), 32, stride=32, pad_lo=3, pad_hi=1, output_padding=31, seed=801),
    P("k32_s1_1d_dil", 1, 4, 6, (40,), 32, stride=1, dilation=3, pad=40, seed=802),
    P("k32_s8_1d", 1, 40, 48, (50,), 32, stride=8, pad=12, seed=803),
    P("k32_s8_1d_bf16", 1, 64, 64, (50,), 32, stride=8, pad=12, dtype="bf16", seed=804),
    P("k32_s32_3d", 1, 2, 3, (2, 3, 2), (32, 2, 3), stride=(32, 2, 1), pad=(5, 0, 1),
      output_padding=(7, 1, 0), seed=805),
    P("k32_grouped_2d", 1, 8, 8, (3, 5), (32, 3), stride=(4, 2), groups=4, pad=(2, 1), seed=806),
]


@pytest.mark.parametrize("p", MAX_KS, ids=lambda p: p.name)
def test_largest_kernel_and_stride_on_every_route(p):
    x, w, b = synth.make_inputs(p)
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    routes = [r for r in supported_routes(p) if r not in (ct.CT_ROUTE_BIAS_FILL, ct.CT_ROUTE_NONE)]
    assert routes, p.name
    for r in routes:
        y = run(p, x, w, b, route=r)
        torch.cuda.synchronize()
        assert_close(p, y, ref, f"route {r}")
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.CT_OK, f"{p.name}: device error word {code:#x}"




# (name, route, problem): y has more than 2^31 elements in each
BIG = [
    ("tc32", ct.CT_ROUTE_TC32_GEMM,
     P("big_tc32", 1, 8, 64, (4_200_000,), 8, stride=8, seed=811)),
    ("tc_bf16", ct.CT_ROUTE_TC_GEMM,
     P("big_tc_bf16", 1, 16, 64, (8_400_000,), 8, stride=4, dtype="bf16", seed=812)),
    ("grouped", ct.CT_ROUTE_GROUPED,
     P("big_grouped", 1, 8, 64, (8_400_000,), 4, stride=4, groups=8, seed=813)),
    ("gather", ct.CT_ROUTE_GATHER,
     P("big_gather", 1, 4, 64, (8_400_000,), 4, stride=4, seed=814)),
]


@pytest.mark.parametrize("name,route,p", BIG, ids=[b[0] for b in BIG])
def test_output_beyond_2_pow_31_elements(name, route, p):
    assert route in supported_routes(p), name
    x, w, b = synth.make_inputs(p)
    y = run(p, x, w, b, route=route)
    torch.cuda.synchronize()
    assert y.numel() > 2 ** 31, (name, y.numel())
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.CT_OK, f"{name}: device error word {code:#x}"
    # sampled outputs: random, the last ones, and those around flat index 2^31
    shape = tuple(y.shape)
    rng = np.random.default_rng(7)
    flat = [rng.integers(0, y.numel(), size=1500)]
    flat.append(np.arange(y.numel() - 64, y.numel()))
    flat.append(np.arange(2 ** 31 - 64, 2 ** 31 + 64))
    flat = np.concatenate(flat)
    idx = np.stack(np.unravel_index(flat, shape), axis=1)
    ref = oracle.points(x, w, b, idx, **p.attrs())
    got = y.reshape(-1)[torch.as_tensor(flat, device=y.device)].to(torch.float64).cpu().numpy()
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL[p.dtype] * scale, f"{name}: max|err| {err:.3e} (max|y| {scale:.3e})"
    del y
    torch.cuda.empty_cache()
