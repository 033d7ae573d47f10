"""Seeded synthetic inputs and the named workloads.

This module only describes problems and draws their inputs.  It holds none
of the transposed convolution's arithmetic (no output shapes, no phase plan),
so both the CUDA path and the fp64 oracle can take their inputs from it.

Inputs are drawn with a CPU ``torch.Generator`` seeded per problem, in fp32,
in the order x, w, bias, then cast to the problem's dtype.  Distributions are
written as ("uniform", lo, hi) or ("normal", mean, variance).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import torch

_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Problem:
    """One forward transposed convolution problem (shapes and attributes)."""
    name: str
    B: int
    C_in: int
    C_out: int
    spatial: Tuple[int, ...]
    k: Tuple[int, ...]
    stride: Tuple[int, ...]
    pad_lo: Tuple[int, ...]
    pad_hi: Tuple[int, ...]
    dilation: Tuple[int, ...]
    output_padding: Tuple[int, ...]
    groups: int = 1
    bias: bool = True
    dtype: str = "f32"
    x_dist: tuple = ("normal", 0.0, 1.0)
    w_dist: tuple = ("normal", 0.0, 1.0)
    b_dist: tuple = ("normal", 0.0, 0.1)
    seed: int = 0

    @property
    def nd(self) -> int:
        return len(self.spatial)

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]

    def attrs(self) -> dict:
        """Keyword attributes shared by the oracle and the binding."""
        return dict(stride=self.stride, pad_lo=self.pad_lo, pad_hi=self.pad_hi,
                    dilation=self.dilation, output_padding=self.output_padding,
                    groups=self.groups)

    def replace(self, **kw) -> "Problem":
        return dataclasses.replace(self, **kw)


def problem(name, B, C_in, C_out, spatial, k, stride=None, pad=None,
            pad_lo=None, pad_hi=None, dilation=None, output_padding=None,
            groups=1, bias=True, dtype="f32", x_dist=("normal", 0.0, 1.0),
            w_dist=("normal", 0.0, 1.0), b_dist=("normal", 0.0, 0.1), seed=0):
    """Build a Problem; scalars broadcast to every spatial axis."""
    nd = len(spatial)

    def vec(v, default):
        if v is None:
            v = default
        if isinstance(v, int):
            v = (v,) * nd
        v = tuple(int(a) for a in v)
        if len(v) != nd:
            raise ValueError(f"expected {nd} values, got {v}")
        return v

    k = vec(k, 1)
    if pad is not None:
        pad_lo = pad if pad_lo is None else pad_lo
        pad_hi = pad if pad_hi is None else pad_hi
    return Problem(name=name, B=B, C_in=C_in, C_out=C_out,
                   spatial=tuple(spatial), k=k, stride=vec(stride, 1),
                   pad_lo=vec(pad_lo, 0), pad_hi=vec(pad_hi, 0),
                   dilation=vec(dilation, 1),
                   output_padding=vec(output_padding, 0), groups=groups,
                   bias=bias, dtype=dtype, x_dist=x_dist, w_dist=w_dist,
                   b_dist=b_dist, seed=seed)


def _draw(gen: torch.Generator, shape, dist) -> torch.Tensor:
    kind = dist[0]
    if kind == "uniform":
        lo, hi = float(dist[1]), float(dist[2])
        return torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    if kind == "normal":
        mean, var = float(dist[1]), float(dist[2])
        return torch.randn(shape, generator=gen, dtype=torch.float32) * math.sqrt(var) + mean
    raise ValueError(f"unknown distribution {dist}")


def make_inputs(p: Problem, seed: Optional[int] = None):
    """Draw (x, w, bias) on the CPU for problem p, cast to p's dtype.

    x: [B, C_in, *spatial]; w: [C_in, C_out/groups, *k]; bias: [C_out] or None.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(p.seed if seed is None else seed)
    x = _draw(gen, (p.B, p.C_in) + tuple(p.spatial), p.x_dist)
    w = _draw(gen, (p.C_in, p.C_out // max(p.groups, 1)) + tuple(p.k), p.w_dist)
    b = _draw(gen, (p.C_out,), p.b_dist) if p.bias else None
    dt = p.torch_dtype
    return x.to(dt), w.to(dt), (b.to(dt) if b is not None else None)


# The five named workloads.  Each draws with seed 1000 + its index.
WORKLOADS: Sequence[Problem] = (
    problem("convT2d_f32_b1_4to3_8x8_k3s2p1op1", 1, 4, 3, (8, 8), 3, stride=2,
            pad=1, output_padding=1, dtype="f32",
            x_dist=("uniform", -1.0, 1.0), w_dist=("uniform", -1.0, 1.0),
            b_dist=("uniform", -1.0, 1.0), seed=1000),
    problem("convT1d_f32_b8_512to256_L2048_k8s4p2", 8, 512, 256, (2048,), 8,
            stride=4, pad=2, dtype="f32", w_dist=("normal", 0.0, 1.0 / (512 * 8)),
            seed=1001),
    problem("convT2d_bf16_b16_256to128_64x64_k4s2p1", 16, 256, 128, (64, 64), 4,
            stride=2, pad=1, dtype="bf16",
            w_dist=("normal", 0.0, 1.0 / (256 * 16)), seed=1002),
    problem("convT2d_f32_b8_256to256_g32_56x56_k3s2p1d2op1", 8, 256, 256,
            (56, 56), 3, stride=2, pad=1, dilation=2, output_padding=1,
            groups=32, dtype="f32", w_dist=("normal", 0.0, 1.0 / (8 * 9)),
            seed=1003),
    problem("convT3d_bf16_b2_128to128_8x64x64_k3s122p1op011", 2, 128, 128,
            (8, 64, 64), 3, stride=(1, 2, 2), pad=1, output_padding=(0, 1, 1),
            dtype="bf16", w_dist=("normal", 0.0, 1.0 / (128 * 27)), seed=1004),
)


def workload(i_or_name) -> Problem:
    if isinstance(i_or_name, int):
        return WORKLOADS[i_or_name]
    for p in WORKLOADS:
        if p.name == i_or_name:
            return p
    raise KeyError(i_or_name)
