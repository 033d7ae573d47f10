"""Pins of the fp64 backward oracle (gradients of ConvTranspose), CPU only.

The SKaiNET pull request "feat(ops): implement convTranspose2d -- CPU kernel,
backward and StableHLO lowering" (#1464) adds the backward as the adjoint of
its scatter-add (input, weight and bias gradients, Summary) and tests it by
finite-difference parity (Tests).  The pins here do not reuse the backward
oracle's code:

- a hand-worked 1-D case in closed form;
- finite differences of the FORWARD oracle (itself pinned elsewhere): the
  loss L = <dy, convT(x, w, b)> is linear in each of x, w and b, so a central
  difference equals the gradient up to rounding, for any step;
- the adjoint identities <convT(x, w), dy> = <x, dx> = <w, dw> and
  <1, dy[:, c]> = db[c];
- float64 torch autograd of conv_transpose{1,2,3}d (a library routine);
- planted mistakes in a copy of the backward oracle, each of which the pins
  must catch.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import _random_problem, _rng, _torch_convT

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "ct_oracle.c")


def _grads(x, w, dy, s, pl, ph, d, op, g):
    return oracle.conv_transpose_backward(x, w, dy, s, pl, ph, d, op, g, threads=2)


def test_hand_case_full_scatter_1d():
    """x = [a, b], w = [p, q], stride 1: y = [ap, aq + bp, bq].  With
    dy = [u, v, z]: dx = [pu + qv, pv + qz], dw = [au + bv, av + bz],
    db = u + v + z."""
    a, b, p, q, u, v, z = 2.0, -3.0, 0.5, 4.0, 1.5, -2.0, 0.25
    x = np.array([[[a, b]]])
    w = np.array([[[p, q]]])
    dy = np.array([[[u, v, z]]])
    dx, dw, db = _grads(x, w, dy, [1], [0], [0], [1], [0], 1)
    assert np.array_equal(dx, np.array([[[p * u + q * v, p * v + q * z]]]))
    assert np.array_equal(dw, np.array([[[a * u + b * v, a * v + b * z]]]))
    assert np.array_equal(db, np.array([u + v + z]))


def test_hand_case_stamp_2d():
    """k2/s2 non-overlapping stamp: y[2i+u, 2j+v] = x[i, j] w[u, v], so
    dx[i, j] = sum_uv w[u, v] dy[2i+u, 2j+v] and dw[u, v] = sum_ij x[i, j]
    dy[2i+u, 2j+v]."""
    r = _rng(3)
    x = r.standard_normal((1, 1, 3, 2))
    w = r.standard_normal((1, 1, 2, 2))
    dy = r.standard_normal((1, 1, 6, 4))
    dx, dw, db = _grads(x, w, dy, [2, 2], [0, 0], [0, 0], [1, 1], [0, 0], 1)
    blocks = dy[0, 0].reshape(3, 2, 2, 2).transpose(0, 2, 1, 3)  # [i, j, u, v]
    assert np.allclose(dx[0, 0], np.einsum("ijuv,uv->ij", blocks, w[0, 0]), rtol=0, atol=1e-14)
    assert np.allclose(dw[0, 0], np.einsum("ijuv,ij->uv", blocks, x[0, 0]), rtol=0, atol=1e-14)
    assert np.isclose(db[0], dy.sum(), rtol=0, atol=1e-13)


def _loss(x, w, b, dy, s, pl, ph, d, op, g):
    y = oracle.conv_transpose(x, w, b, s, pl, ph, d, op, g, threads=2)
    return float(np.sum(y * dy))


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_finite_differences_of_the_forward_oracle(nd):
    r = _rng(40 + nd)
    for _ in range(8):
        x, w, bias, s, pl, ph, d, op, g = _random_problem(r, nd)
        if bias is None:
            bias = np.zeros(w.shape[1] * g)
        O = oracle.out_shape(x.shape[2:], w.shape[2:], s, pl, ph, d, op)
        dy = r.standard_normal((x.shape[0], w.shape[1] * g) + O)
        dx, dw, db = _grads(x, w, dy, s, pl, ph, d, op, g)
        h = 0.5
        for arr, grad, which in ((x, dx, 0), (w, dw, 1), (bias, db, 2)):
            flat = arr.reshape(-1)
            for e in r.choice(flat.size, size=min(6, flat.size), replace=False):
                args = [x, w, bias]
                plus, minus = flat.copy(), flat.copy()
                plus[e] += h
                minus[e] -= h
                args[which] = plus.reshape(arr.shape)
                lp = _loss(*args, dy, s, pl, ph, d, op, g)
                args[which] = minus.reshape(arr.shape)
                lm = _loss(*args, dy, s, pl, ph, d, op, g)
                fd = (lp - lm) / (2 * h)
                gv = grad.reshape(-1)[e]
                assert abs(fd - gv) <= 1e-11 * max(1.0, abs(gv)), (which, fd, gv)


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_adjoint_identities(nd):
    r = _rng(50 + nd)
    for _ in range(25):
        x, w, _, s, pl, ph, d, op, g = _random_problem(r, nd)
        y = oracle.conv_transpose(x, w, None, s, pl, ph, d, op, g, threads=2)
        dy = r.standard_normal(y.shape)
        dx, dw, db = _grads(x, w, dy, s, pl, ph, d, op, g)
        ip = float(np.sum(y * dy))
        scale = max(1.0, float(np.sum(np.abs(y * dy))))
        assert abs(ip - float(np.sum(x * dx))) <= 1e-12 * scale
        assert abs(ip - float(np.sum(w * dw))) <= 1e-12 * scale
        assert np.allclose(db, dy.sum(axis=tuple([0] + list(range(2, dy.ndim)))),
                           rtol=1e-13, atol=1e-12)


_CONVT = {1: torch.nn.functional.conv_transpose1d, 2: torch.nn.functional.conv_transpose2d,
          3: torch.nn.functional.conv_transpose3d}


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_matches_torch_autograd_f64(nd):
    """Symmetric pads (torch's own convention); asymmetric pads are covered by
    the finite differences and the adjoint identities."""
    r = _rng(60 + nd)
    for _ in range(20):
        x, w, bias, s, pl, ph, d, op, g = _random_problem(r, nd)
        pl = ph = [min(a, b) for a, b in zip(pl, ph)]
        O = oracle.out_shape(x.shape[2:], w.shape[2:], s, pl, ph, d, op)
        if min(O) < 1:
            continue
        dy = r.standard_normal((x.shape[0], w.shape[1] * g) + O)
        xt = torch.from_numpy(x).requires_grad_(True)
        wt = torch.from_numpy(w).requires_grad_(True)
        bt = torch.zeros(w.shape[1] * g, dtype=torch.float64, requires_grad=True)
        yt = _CONVT[nd](xt, wt, bt, stride=tuple(s), padding=tuple(pl), output_padding=tuple(op),
                        groups=g, dilation=tuple(d))
        yt.backward(torch.from_numpy(dy))
        dx, dw, db = _grads(x, w, dy, s, pl, ph, d, op, g)
        assert np.allclose(dx, xt.grad.numpy(), rtol=1e-12, atol=1e-12)
        assert np.allclose(dw, wt.grad.numpy(), rtol=1e-12, atol=1e-12)
        assert np.allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_gradients_not_requested_are_skipped():
    r = _rng(70)
    x, w, _, s, pl, ph, d, op, g = _random_problem(r, 2)
    O = oracle.out_shape(x.shape[2:], w.shape[2:], s, pl, ph, d, op)
    dy = r.standard_normal((x.shape[0], w.shape[1] * g) + O)
    dx, dw, db = oracle.conv_transpose_backward(x, w, dy, s, pl, ph, d, op, g, need=("dw",))
    assert dx is None and db is None and dw is not None
    full = _grads(x, w, dy, s, pl, ph, d, op, g)
    assert np.array_equal(dw, full[1])


# ---------------------------------------------------------------------------
# planted mistakes in the backward oracle (the section after its marker)
# ---------------------------------------------------------------------------

MARK = " * Backward pass (gradients), in fp64"
BMUTANTS = [
    ("dx pad sign", "const int64_t o2 = i2 * p->S[2] - p->PL[2] + t2 * p->DL[2];\n"
     "                        if (o2 < 0 || o2 >= p->O[2]) continue;\n"
     "                        dxr[i2]",
     "const int64_t o2 = i2 * p->S[2] + p->PL[2] + t2 * p->DL[2];\n"
     "                        if (o2 < 0 || o2 >= p->O[2]) continue;\n"
     "                        dxr[i2]"),
    ("dx transposed weight", "const double* ws = j->w + (ic * Cog + oc_g) * Kn;",
     "const double* ws = j->w + (oc_g * p->C_in + ic) * Kn;"),
    ("dw dropped dilation", "const int64_t o1 = i1 * p->S[1] - p->PL[1] + t1 * p->DL[1];\n"
     "                        if (o1 < 0 || o1 >= p->O[1]) continue;\n"
     "                        const double* xr",
     "const int64_t o1 = i1 * p->S[1] - p->PL[1] + t1;\n"
     "                        if (o1 < 0 || o1 >= p->O[1]) continue;\n"
     "                        const double* xr"),
    ("dw one batch only", "for (int64_t b = 0; b < p->B; ++b) {\n                const double* xs",
     "for (int64_t b = 0; b < 1; ++b) {\n                const double* xs"),
    ("dw tap order reversed",
     "j->dw[(ic * Cog + oc_g) * Kn + (t0 * p->K[1] + t1) * p->K[2] + t2] = acc;",
     "j->dw[(ic * Cog + oc_g) * Kn + (t0 * p->K[1] + t1) * p->K[2] + (p->K[2] - 1 - t2)] = acc;"),
    ("db first batch only", "for (int64_t b = 0; b < p->B; ++b) {\n        const double* dys",
     "for (int64_t b = 0; b < 1; ++b) {\n        const double* dys"),
    ("dx group index", "const int64_t g = ic / Cig;\n    const int64_t In = p->I[0] * p->I[1] * p->I[2];\n"
     "    const int64_t On = p->O[0] * p->O[1] * p->O[2];\n    const int64_t Kn = p->K[0] * p->K[1] * p->K[2];\n"
     "    double* dxs",
     "const int64_t g = 0;\n    const int64_t In = p->I[0] * p->I[1] * p->I[2];\n"
     "    const int64_t On = p->O[0] * p->O[1] * p->O[2];\n    const int64_t Kn = p->K[0] * p->K[1] * p->K[2];\n"
     "    double* dxs"),
]

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def _build_backward(tmp_path, text, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(text)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                           str(so), str(c), "-lm"])
    f = ctypes.CDLL(str(so)).oracle_conv_transpose_backward_f64
    f.restype = ctypes.c_int
    f.argtypes = [_f64p] * 6 + [ctypes.c_int] + [ctypes.c_int64] * 4 + [_i64p] * 7 + [ctypes.c_int]
    return f


def _backward_disagrees(f):
    """Pins against torch autograd in float64, on symmetric-pad problems."""
    r = _rng(91)
    for nd in (1, 2, 3):
        for _ in range(12):
            x, w, _, s, pl, ph, d, op, g = _random_problem(r, nd)
            pl = ph = [min(a, b) for a, b in zip(pl, ph)]
            ref_y = _torch_convT(x, w, None, s, pl, ph, d, op, g)
            dy = r.standard_normal(ref_y.shape)
            xt = torch.from_numpy(x).requires_grad_(True)
            wt = torch.from_numpy(w).requires_grad_(True)
            bt = torch.zeros(w.shape[1] * g, dtype=torch.float64, requires_grad=True)
            _CONVT[nd](xt, wt, bt, stride=tuple(s), padding=tuple(pl), output_padding=tuple(op),
                       groups=g, dilation=tuple(d)).backward(torch.from_numpy(dy))
            dx, dw, db = np.zeros_like(x), np.zeros_like(w), np.zeros(w.shape[1] * g)
            arrs = [np.ascontiguousarray(np.array(v, dtype=np.int64))
                    for v in (x.shape[2:], w.shape[2:], s, pl, ph, d, op)]
            pp = lambda a: a.ctypes.data_as(_f64p)
            xc, wc, dyc = (np.ascontiguousarray(a) for a in (x, w, dy))
            rc = f(pp(xc), pp(wc), pp(dyc), pp(dx), pp(dw), pp(db), nd, x.shape[0], x.shape[1],
                   w.shape[1] * g, g, *[a.ctypes.data_as(_i64p) for a in arrs], 1)
            if rc != 0:
                return True
            for got, ref in ((dx, xt.grad), (dw, wt.grad), (db, bt.grad)):
                if not np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12):
                    return True
    return False


def test_unmutated_backward_copy_agrees(tmp_path):
    assert not _backward_disagrees(_build_backward(tmp_path, open(SRC).read(), "orig"))


@pytest.mark.parametrize("name,old,new", BMUTANTS, ids=[m[0] for m in BMUTANTS])
def test_backward_mutant_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    head, tail = text.split(MARK, 1)
    assert tail.count(old) == 1, f"mutation site for '{name}' not unique"
    f = _build_backward(tmp_path, head + MARK + tail.replace(old, new), "mut")
    assert _backward_disagrees(f), f"planted mistake '{name}' was not caught"
