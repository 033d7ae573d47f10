"""Planted mistakes: each mutant of the oracle must fail the pins.

A copy of ct_oracle.c is edited on the CPU (one plausible mistake per copy:
a wrong sign, a dropped term, a transposed operand, a wrong group index),
compiled into a temporary library and run against the same library-routine
pin as test_oracle_pins (torch conv_transposeNd in float64).  The test passes
when every mutant disagrees with the pin somewhere; the real oracle agrees.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from test_oracle_pins import _random_problem, _rng, _torch_convT

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "ct_oracle.c")

# (name, text in the scatter, replacement)
MUTANTS = [
    ("pad sign", "o2 = i2 * p->S[2] - p->PL[2]", "o2 = i2 * p->S[2] + p->PL[2]"),
    ("dropped dilation", "t1 * p->DL[1];\n                    if (o1",
     "t1;\n                    if (o1"),
    ("transposed weight operand", "ws = job->w + (ic * Cog + oc_g) * Kn",
     "ws = job->w + (oc_g * p->C_in + ic) * Kn"),
    ("dropped bias", "ys[o] = init;", "ys[o] = 0.0;"),
    ("group index", "const int64_t ic = g * Cig + ic_g;\n        const double* xs",
     "const int64_t ic = ic_g;\n        const double* xs"),
    ("output padding ignored", "+ DL * (K - 1) + OP + 1", "+ DL * (K - 1) + 1"),
    ("stride on the wrong axis", "o0 = i0 * p->S[0]", "o0 = i0 * p->S[2]"),
    ("tap order reversed", "ws[(t0 * p->K[1] + t1) * p->K[2] + t2]",
     "ws[(t0 * p->K[1] + t1) * p->K[2] + (p->K[2] - 1 - t2)]"),
]

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def _build(tmp_path, text, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(text)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared",
                           "-pthread", "-o", str(so), str(c), "-lm"])
    lib = ctypes.CDLL(str(so))
    f = lib.oracle_conv_transpose_f64
    f.restype = ctypes.c_int
    f.argtypes = ([_f64p] * 4 + [ctypes.c_int] + [ctypes.c_int64] * 4
                  + [_i64p] * 7 + [ctypes.c_int])
    return f


def _run(f, x, w, bias, s, pl, ph, d, op, g, O):
    nd = x.ndim - 2
    C_out = w.shape[1] * g
    y = np.zeros((x.shape[0], C_out) + tuple(O))
    arrs = [np.ascontiguousarray(np.array(v, dtype=np.int64))
            for v in (x.shape[2:], w.shape[2:], s, pl, ph, d, op)]
    p = lambda a: None if a is None else np.ascontiguousarray(a).ctypes.data_as(_f64p)
    xc, wc = np.ascontiguousarray(x), np.ascontiguousarray(w)
    bc = None if bias is None else np.ascontiguousarray(bias)
    rc = f(p(xc), p(wc), p(bc), y.ctypes.data_as(_f64p), nd, x.shape[0],
           x.shape[1], C_out, g, *[a.ctypes.data_as(_i64p) for a in arrs], 1)
    return rc, y


def _disagrees(f):
    r = _rng(77)
    for nd in (1, 2, 3):
        for _ in range(30):
            x, w, bias, s, pl, ph, d, op, g = _random_problem(r, nd)
            ref = _torch_convT(x, w, bias, s, pl, ph, d, op, g)
            rc, y = _run(f, x, w, bias, s, pl, ph, d, op, g, ref.shape[2:])
            if rc != 0 or not np.allclose(y, ref, rtol=1e-12, atol=1e-12):
                return True
    return False


def test_unmutated_copy_agrees(tmp_path):
    f = _build(tmp_path, open(SRC).read(), "orig")
    assert not _disagrees(f)


# the forward part of the file; the backward oracle after this marker has
# its own mutants (test_oracle_backward_pins)
MARK = " * Backward pass (gradients), in fp64"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    head, tail = text.split(MARK, 1)
    assert head.count(old) == 1, f"mutation site for '{name}' not unique"
    f = _build(tmp_path, head.replace(old, new) + MARK + tail, "mut")
    assert _disagrees(f), f"planted mistake '{name}' was not caught"
