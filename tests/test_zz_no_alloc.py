"""The entry point that allocates no device memory.

ct_conv_transpose_nd_noalloc is for callers that may not call cudaMalloc
where they run the convolution (graph capture that forbids allocation,
engine plugins limited to engine-provided memory, frameworks that own the
memory budget, real-time code).  It keeps its scratch in one static device
array.  These checks call it through the C ABI and compare it with the
regular entry point, ct_conv_transpose_nd, within the tolerance the parity
tests use, over two calls in a row on different problems (so the second
call starts from the scratch contents the first one left).  This file is
collected last so that a stop-at-first-failure run has run everything else.
"""
import numpy as np
import pytest
import torch

import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import TOL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transposed_convolution_convtranspose1_gb300 import _build
    _build.build_library()
    ct.lib()
    yield


def _outputs(p):
    x, w, b = to_device(*synth.make_inputs(p))
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    y_ref = torch.empty((p.B, p.C_out) + O, dtype=p.torch_dtype, device="cuda")
    y_na = torch.full_like(y_ref, float("nan"))
    a = dict(stride=p.stride, pad_lo=p.pad_lo, pad_hi=p.pad_hi, dilation=p.dilation,
             output_padding=p.output_padding, groups=p.groups)
    ct.ct_conv_transpose_nd(x, w, b, y_ref, None, **a)
    ct.ct_conv_transpose_nd_noalloc(x, w, b, y_na, **a)
    torch.cuda.synchronize()
    return y_ref, y_na


def _check(p, y_ref, y_na):
    ref = y_ref.double()
    err = float((y_na.double() - ref).abs().max())
    bound = TOL[p.dtype] * float(ref.abs().max())
    assert err <= bound, f"{p.name}: max|err| {err:.3e} > {bound:.3e}"


def test_two_calls_in_a_row_match_the_regular_entry_point():
    first = synth.workload(2)    # bf16 2-D, tensor-core route, 34.6 MB of scratch
    second = synth.workload(4)   # bf16 3-D, tensor-core route, different scratch layout
    for p in (first, second):
        need = ct.ct_conv_transpose_workspace_bytes(
            p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
            p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))
        assert 0 < need <= ct.CT_NOALLOC_SCRATCH_BYTES
        y_ref, y_na = _outputs(p)
        _check(p, y_ref, y_na)


def test_route_without_scratch_also_runs():
    p = synth.workload(0)          # fp32 problem on a route that needs no scratch
    y_ref, y_na = _outputs(p)
    _check(p, y_ref, y_na)


def test_problem_larger_than_the_scratch_is_rejected():
    p = synth.problem("too_big", 1, 64, 16, (1024, 1024), 2, stride=2, dtype="bf16", seed=5)
    need = ct.ct_conv_transpose_workspace_bytes(
        p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
        p.output_padding, p.groups, ct.dtype_code(p.torch_dtype))
    assert need > ct.CT_NOALLOC_SCRATCH_BYTES
    x = torch.zeros((1, 64, 1024, 1024), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((64, 16, 2, 2), dtype=torch.bfloat16, device="cuda")
    y = torch.full((1, 16, 2048, 2048), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ct.CtError) as e:
        ct.ct_conv_transpose_nd_noalloc(x, w, None, y, stride=2)
    assert e.value.status == ct.ct.CT_ERR_WORKSPACE
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
