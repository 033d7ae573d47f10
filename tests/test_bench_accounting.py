"""bench.py's work accounting against the oracle, CPU only.

FLOP in every bench line is 2 x valid_macs(p): the multiply-adds whose
product lands inside the output.  With x and w all ones and no bias, each
output of the fp64 oracle counts the products that land on it, so the
oracle's total is that number, computed by the scatter itself rather than by
bench's per-axis formula.  The byte count is checked against the tensors'
own sizes.
"""
import importlib.util
import os

import numpy as np
import pytest
import torch

import oracle
from transposed_convolution_convtranspose1_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _grid():
    r = np.random.default_rng(77)
    out = []
    for n in range(24):
        nd = int(r.integers(1, 4))
        G = int(r.choice([1, 2, 3]))
        spatial, k, s, d, pl, ph, op = [], [], [], [], [], [], []
        for _ in range(nd):
            spatial.append(int(r.integers(1, 7)))
            k.append(int(r.integers(1, 5)))
            s.append(int(r.integers(1, 4)))
            d.append(int(r.integers(1, 3)))
            op.append(int(r.integers(0, max(s[-1], d[-1]))))
            while True:
                a, b = int(r.integers(0, 4)), int(r.integers(0, 4))
                if (spatial[-1] - 1) * s[-1] - a - b + d[-1] * (k[-1] - 1) + op[-1] + 1 >= 1:
                    break
            pl.append(a)
            ph.append(b)
        out.append(synth.problem(f"acct{n}", int(r.integers(1, 3)), G * int(r.integers(1, 4)),
                                 G * int(r.integers(1, 4)), tuple(spatial), tuple(k),
                                 stride=tuple(s), pad_lo=tuple(pl), pad_hi=tuple(ph),
                                 dilation=tuple(d), output_padding=tuple(op), groups=G,
                                 bias=bool(n % 2)))
    return out


@pytest.mark.parametrize("p", _grid(), ids=lambda p: p.name)
def test_valid_macs_is_the_scatter_count(bench, p):
    x = torch.ones((p.B, p.C_in) + p.spatial, dtype=torch.float64)
    w = torch.ones((p.C_in, p.C_out // p.groups) + p.k, dtype=torch.float64)
    y = oracle.conv_transpose(x, w, None, **p.attrs())
    assert float(y.sum()) == bench.valid_macs(p)


@pytest.mark.parametrize("i", range(5))
def test_alg_bytes_of_the_workloads(bench, i):
    p = synth.workload(i)
    x, w, b = synth.make_inputs(p.replace(B=1)) if i else synth.make_inputs(p)
    eb = x.element_size()
    O = bench.out_shape(p)
    want = (p.B * p.C_in * int(np.prod(p.spatial)) + w.numel() + (p.C_out if p.bias else 0)
            + p.B * p.C_out * int(np.prod(O))) * eb
    assert bench.alg_bytes(p) == want
