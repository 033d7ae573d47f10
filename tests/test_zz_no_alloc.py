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
import ctypes
import glob
import os

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


def _cudart():
    """The CUDA runtime as a shared library (for the memory-pool counters)."""
    cands = ["/usr/local/cuda/lib64/libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"]
    cands += glob.glob(os.path.join(os.path.dirname(os.path.dirname(torch.__file__)), "nvidia",
                                    "*", "lib", "libcudart.so*"))
    for c in cands:
        if os.path.exists(c):
            try:
                return ctypes.CDLL(c)
            except OSError:
                pass
    pytest.skip("no shared CUDA runtime library to read the memory-pool counters")


CUDA_MEMPOOL_ATTR_USED_MEM_HIGH = 8  # cudaMemPoolAttrUsedMemHigh


def test_the_call_takes_no_stream_ordered_memory():
    """The regular entry point without a workspace takes its scratch from the
    device's default memory pool (cudaMallocAsync); the no-allocation entry
    point must not.  The pool's high-water mark of used memory, reset to 0
    before each call, tells which one allocated."""
    rt = _cudart()
    dev = torch.cuda.current_device()
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0

    def used_high_after(call):
        zero = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, CUDA_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(zero)) == 0
        call()
        torch.cuda.synchronize()
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, CUDA_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(v)) == 0
        return v.value

    p = synth.workload(2)  # a route that needs scratch
    x, w, b = to_device(*synth.make_inputs(p))
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    y = torch.empty((p.B, p.C_out) + O, dtype=p.torch_dtype, device="cuda")
    a = dict(stride=p.stride, pad_lo=p.pad_lo, pad_hi=p.pad_hi, dilation=p.dilation,
             output_padding=p.output_padding, groups=p.groups)
    ct.ct_conv_transpose_nd_noalloc(x, w, b, y, **a)  # first call: address look-up
    torch.cuda.synchronize()
    # the check sees an allocation when there is one
    assert used_high_after(lambda: ct.ct_conv_transpose_nd(x, w, b, y, None, **a)) > 0
    assert used_high_after(lambda: ct.ct_conv_transpose_nd_noalloc(x, w, b, y, **a)) == 0
