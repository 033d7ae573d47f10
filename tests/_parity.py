"""Helpers for the GPU parity tests: run the CUDA path, compare with the oracle.

Tolerance (max-norm, relative to the largest oracle output):
    fp32 in/out                : max|y - y_oracle| <= 1e-5 * max|y_oracle|
    bf16/fp16 in/out, fp32 acc : max|y - y_oracle| <= 1e-2 * max|y_oracle|
Shapes must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import transposed_convolution_convtranspose1_gb300 as ct
from transposed_convolution_convtranspose1_gb300 import synth

TOL = {"f32": 1e-5, "f16": 1e-2, "bf16": 1e-2}


def to_device(x, w, b, dev="cuda"):
    return x.to(dev), w.to(dev), (None if b is None else b.to(dev))


def run(p: synth.Problem, x, w, b, route=ct.CT_ROUTE_AUTO, workspace=None, stream=None):
    xd, wd, bd = to_device(x, w, b)
    O = ct.ct_conv_transpose_out_shape(p.spatial, p.k, p.stride, p.pad_lo, p.pad_hi,
                                       p.dilation, p.output_padding)
    y = torch.empty((p.B, p.C_out) + O, dtype=p.torch_dtype, device="cuda")
    ct.ct_conv_transpose_nd(xd, wd, bd, y, workspace, p.stride, p.pad_lo, p.pad_hi, p.dilation,
                            p.output_padding, p.groups, route, stream)
    return y


def max_err(y: torch.Tensor, ref: np.ndarray):
    got = y.detach().to(torch.float64).cpu().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    return err, scale


def assert_close(p, y, ref, what=""):
    err, scale = max_err(y, ref)
    bound = TOL[p.dtype] * scale
    assert err <= bound, f"{p.name} {what}: max|err| = {err:.3e} > {bound:.3e} (max|y| {scale:.3e})"
    return err, scale


def check_full(p, route=ct.CT_ROUTE_AUTO, seed=None):
    x, w, b = synth.make_inputs(p, seed)
    y = run(p, x, w, b, route)
    torch.cuda.synchronize()
    ref = oracle.conv_transpose(x, w, b, **p.attrs())
    return assert_close(p, y, ref, f"route {route}")


def supported_routes(p):
    """Routes (besides AUTO) that can run problem p on this device."""
    out = []
    for r in (ct.CT_ROUTE_GATHER, ct.CT_ROUTE_GROUPED, ct.CT_ROUTE_SIMT_GEMM,
              ct.CT_ROUTE_TC_GEMM, ct.CT_ROUTE_TC32_GEMM, ct.CT_ROUTE_BIAS_FILL,
              ct.CT_ROUTE_NONE):
        try:
            ct.ct_conv_transpose_workspace_bytes(p.B, p.C_in, p.C_out, p.spatial, p.k, p.stride,
                                                 p.pad_lo, p.pad_hi, p.dilation,
                                                 p.output_padding, p.groups,
                                                 ct.dtype_code(p.torch_dtype), route=r)
            out.append(r)
        except ct.CtError as e:
            assert e.status == ct.ct.CT_ERR_ROUTE
    return out


def sample_indices(shape, n, rng):
    """n random output coordinates plus every corner of the output box."""
    idx = [rng.integers(0, s, size=n) for s in shape]
    idx = np.stack(idx, axis=1)
    corners = np.array(np.meshgrid(*[[0, s - 1] for s in shape], indexing="ij")).reshape(
        len(shape), -1).T
    return np.concatenate([idx, corners], axis=0)
