"""The bounded device-side waits give up cleanly and say so.

Every kernel that waits on an asynchronous copy or MMA bounds the wait.  A
limit of 0 (ct_set_wait_limit_ns) makes each wait that is reached give up at
once, as if what it waits for never arrived.  On each kernel that waits --
the bf16 and the error-compensated TF32 tensor-core GEMMs, the grouped warp
pairs, the grouped TMA kernel and the backward pass's small-group dw kernel
(fp32 rows staged by bulk copies) -- the call must then return, the
kernels must stop after draining what they had issued (no hang, no fault),
ct_device_status must report CT_ERR_DEVICE_TIMEOUT with the giving-up role's
bit, and with the default limit restored the same call must match the fp64
oracle with a clean status word.  This is the pull request's rule that bad
states fail loudly (SKaiNET "feat(ops): implement convTranspose2d", Summary)
applied to device waits.
"""
import pytest
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth
from _parity import assert_close, run

pytestmark = pytest.mark.gpu

P = synth.problem

# (problem, kernel that must run it, error bits its give-up must set)
CASES = [
    (P("wl_bf16", 2, 64, 32, (9, 12), 4, stride=2, pad=1, dtype="bf16", seed=7),
     "tc_phase_gemm", 0x1 | 0x2),
    (P("wl_tf32", 2, 64, 40, (37,), 8, stride=4, pad=2, seed=601), "tc32_phase_gemm", 0x1 | 0x2),
    (P("wl_grouped_warp", 1, 16, 16, (20, 32), 3, stride=2, pad=1, dilation=2, output_padding=1,
       groups=2, seed=712), "grouped_warp_kernel", 0x20 | 0x40),
    (P("wl_grouped_tma_3d", 1, 16, 16, (5, 12, 12), (4, 3, 3), stride=(1, 2, 2), pad=1,
       output_padding=(0, 1, 1), groups=2, seed=720), "grouped_tma_kernel", 0x10),
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
    ct.ct_set_wait_limit_ns(ct.CT_WAIT_LIMIT_DEFAULT_NS)
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.CT_OK, f"device error word set: {code:#x}"


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_wait_that_gives_up_is_reported_and_the_next_call_is_correct(case):
    p, kernel, bits = case
    assert ct.ct_conv_transpose_kernel(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride, p.pad_lo,
                                       p.pad_hi, p.dilation, p.output_padding, p.groups,
                                       ct.dtype_code(p.torch_dtype)) == kernel
    x, w, b = synth.make_inputs(p)
    prev = ct.ct_set_wait_limit_ns(0)
    try:
        run(p, x, w, b)  # returns: the launches themselves succeed
    finally:
        assert ct.ct_set_wait_limit_ns(prev) == 0
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.ct.CT_ERR_DEVICE_TIMEOUT, (rc, hex(code))
    assert code & bits == bits, f"{kernel}: word {code:#x} lacks bits {bits:#x}"
    assert code & 0x8 == 0, "a drain after the give-up ran out"
    # the word is cleared and the device is healthy: a normal call matches the oracle
    assert ct.ct_device_status(clear=True) == (ct.CT_OK, 0)
    y = run(p, x, w, b)
    torch.cuda.synchronize()
    assert_close(p, y, oracle.conv_transpose(x, w, b, **p.attrs()), "after the give-up")
    assert ct.ct_device_status(clear=True) == (ct.CT_OK, 0)


def test_default_limit_is_restored():
    prev = ct.ct_set_wait_limit_ns(ct.CT_WAIT_LIMIT_DEFAULT_NS)
    assert prev == ct.CT_WAIT_LIMIT_DEFAULT_NS


def test_grouped_dw_copy_wait_gives_up_and_the_next_call_is_correct():
    """The small-group dw kernel's row-copy staged bands: with a limit of 0 the
    first band's wait gives up (bit 128), the block drains the copies it
    issued and writes nothing; the backward call returns.  With the default
    limit the same call matches the oracle's dw."""
    p = P("wl_dw_grouped", 2, 16, 16, (13, 16), 3, stride=2, pad=1, output_padding=1, groups=2,
          seed=730)
    x, w, _ = synth.make_inputs(p)
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi, p.dilation,
                                       p.output_padding)
    dy = torch.randn((p.B, p.C_out) + tuple(O), generator=torch.Generator().manual_seed(5))
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()

    def dw_call():
        dw = torch.full_like(wd, float("nan"))
        ct.ct_conv_transpose_backward_nd(xd, wd, dyd, None, dw, None, None, p.stride, p.pad_lo,
                                         p.pad_hi, p.dilation, p.output_padding, p.groups)
        return dw

    prev = ct.ct_set_wait_limit_ns(0)
    try:
        dw_call()
    finally:
        assert ct.ct_set_wait_limit_ns(prev) == 0
    rc, code = ct.ct_device_status(clear=True)
    assert rc == ct.ct.CT_ERR_DEVICE_TIMEOUT, (rc, hex(code))
    assert code & 0x80, f"word {code:#x} lacks the dw copy bit 0x80"
    assert code & 0x8 == 0, "a drain after the give-up ran out"
    dw = dw_call()
    torch.cuda.synchronize()
    assert ct.ct_device_status(clear=True) == (ct.CT_OK, 0)
    _, rdw, _ = oracle.conv_transpose_backward(x, w, dy, **p.attrs(), need=("dw",))
    ref = torch.from_numpy(rdw)
    err = float((dw.cpu().double() - ref).abs().max())
    assert err <= 1e-5 * float(ref.abs().max())
