"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

None of these re-types the oracle's own formula.  They check it against
- output shapes the pages and workloads state (tests/golden/out_shapes.json),
- the two hand-computed cases named in the SKaiNET pull request's test list
  (kernel 2 at stride 1, where every tap overlaps its neighbours, and
  kernel 2 at stride 2, where the taps tile the output without overlap), in
  closed form,
- library routines: scipy's full N-D convolution (stride 1, no padding),
  torch.nn.functional.conv_transposeNd and convNd in float64,
- the forward-convolution equivalence the pages use (input dilated by the
  stride, taps reversed, pads dilation*(k-1) - pad; ONNX page
  ncdhw3d_implicit_sgmat, SKaiNET StableHLO lowering, NKI conv3d_transpose),
- the adjoint identity <convT(x), y> = <x, conv(y)> behind the SKaiNET
  backward pass,
- linearity, the bias shift, the 1x1 plain-GEMM case, thread invariance, and
  the agreement of point evaluation with the full scatter.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "out_shapes.json")


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# output shapes
# --------------------------------------------------------------------------

def test_out_shapes_golden():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) == 6
    for c in cases:
        nd = len(c["x"]) - 2
        got = oracle.out_shape(c["x"][2:], c["w"][2:], c["stride"], c["pad_lo"],
                               c["pad_hi"], c["dilation"], c["output_padding"])
        C_out = c["w"][1] * c["groups"]
        assert (c["x"][0], C_out) + got == tuple(c["y"]), c["source"]
        assert len(got) == nd


def test_out_shape_hand_table():
    # (I, k, s, pad_lo, pad_hi, d, op) -> O, each worked by hand.
    table = [
        ((2,), (2,), (1,), (0,), (0,), (1,), (0,), (3,)),   # k2/s1 full scatter
        ((2,), (2,), (2,), (0,), (0,), (1,), (0,), (4,)),   # k2/s2 stamp
        ((5,), (3,), (1,), (1,), (1,), (1,), (0,), (5,)),   # "same" transposed conv
        ((5,), (3,), (2,), (0,), (2,), (1,), (1,), (10,)),  # asymmetric pads + op
        ((4,), (3,), (3,), (0,), (0,), (2,), (1,), (15,)),  # dilation 2, op 1
        ((1,), (1,), (7,), (0,), (0,), (1,), (6,), (7,)),   # op up to s-1
        ((3, 4), (2, 3), (2, 1), (1, 0), (0, 2), (1, 2), (1, 0), (6, 6)),
    ]
    for I, k, s, pl, ph, d, op, O in table:
        assert oracle.out_shape(I, k, s, pl, ph, d, op) == O


def test_out_shape_rejects_empty_output():
    with pytest.raises(ValueError):
        oracle.out_shape((1,), (1,), (1,), (1,), (0,), (1,), (0,))  # O = 0
    with pytest.raises(ValueError):
        oracle.out_shape((2,), (2,), (1,), (2,), (2,), (1,), (0,))  # O = -1


# --------------------------------------------------------------------------
# hand-computed cases (SKaiNET test list: k2/s1 full scatter, k2/s2 stamp)
# --------------------------------------------------------------------------

def test_k2s1_full_scatter_1d_closed_form():
    a, b, p, q = 0.75, -1.25, 2.5, 0.375
    x = np.array([[[a, b]]])
    w = np.array([[[p, q]]])
    y = oracle.conv_transpose(x, w)
    np.testing.assert_array_equal(y[0, 0], [a * p, a * q + b * p, b * q])


def test_k2s1_full_scatter_2d_is_full_convolution():
    scipy_signal = pytest.importorskip("scipy.signal")
    r = _rng(1)
    x = r.standard_normal((1, 1, 5, 4))
    w = r.standard_normal((1, 1, 2, 2))
    y = oracle.conv_transpose(x, w)
    ref = scipy_signal.convolve(x[0, 0], w[0, 0], mode="full", method="direct")
    np.testing.assert_allclose(y[0, 0], ref, rtol=0, atol=1e-13)


def test_stride1_nopad_equals_full_nd_convolution_multichannel():
    # convT with s=1, p=0, d=1 is, per (ic, oc) pair, the full convolution of
    # the input plane with the kernel, summed over ic.
    scipy_signal = pytest.importorskip("scipy.signal")
    r = _rng(2)
    for nd in (1, 2, 3):
        sp = (4, 3, 5)[:nd]
        k = (3, 2, 2)[:nd]
        x = r.standard_normal((2, 3) + sp)
        w = r.standard_normal((3, 2) + k)
        bias = r.standard_normal(2)
        y = oracle.conv_transpose(x, w, bias)
        for b in range(2):
            for oc in range(2):
                ref = sum(scipy_signal.convolve(x[b, ic], w[ic, oc], mode="full",
                                                method="direct") for ic in range(3))
                np.testing.assert_allclose(y[b, oc], ref + bias[oc], atol=1e-12)


def test_k2s2_non_overlapping_stamp_exact():
    r = _rng(3)
    x = r.standard_normal((1, 1, 3, 4))
    w = r.standard_normal((1, 1, 2, 2))
    y = oracle.conv_transpose(x, w, stride=(2, 2))
    assert y.shape == (1, 1, 6, 8)
    for i in range(3):
        for j in range(4):
            for u in range(2):
                for v in range(2):
                    assert y[0, 0, 2 * i + u, 2 * j + v] == x[0, 0, i, j] * w[0, 0, u, v]


# --------------------------------------------------------------------------
# library special case: torch conv_transposeNd in float64
# --------------------------------------------------------------------------

_CONVT = {1: F.conv_transpose1d, 2: F.conv_transpose2d, 3: F.conv_transpose3d}
_CONV = {1: F.conv1d, 2: F.conv2d, 3: F.conv3d}


def _torch_convT(x, w, bias, s, pl, ph, d, op, g):
    """torch conv_transpose with symmetric pad min(pl, ph), then a crop.

    A smaller pad on one side only adds output positions on that side, so the
    asymmetric result is a window of the symmetric one.
    """
    nd = x.ndim - 2
    pm = [min(a, b) for a, b in zip(pl, ph)]
    yt = _CONVT[nd](torch.from_numpy(x), torch.from_numpy(w),
                    None if bias is None else torch.from_numpy(bias),
                    stride=tuple(s), padding=tuple(pm), output_padding=tuple(op),
                    groups=g, dilation=tuple(d)).numpy()
    sl = [slice(None), slice(None)]
    for a in range(nd):
        lo = pl[a] - pm[a]
        hi = yt.shape[2 + a] - (ph[a] - pm[a])
        sl.append(slice(lo, hi))
    return yt[tuple(sl)]


def _random_problem(r, nd):
    g = int(r.choice([1, 1, 2, 3]))
    Cig = int(r.integers(1, 4))
    Cog = int(r.integers(1, 4))
    B = int(r.integers(1, 3))
    I, k, s, pl, ph, d, op = [], [], [], [], [], [], []
    for _ in range(nd):
        I.append(int(r.integers(1, 6)))
        k.append(int(r.integers(1, 5)))
        s.append(int(r.integers(1, 4)))
        d.append(int(r.integers(1, 4)))
        op.append(int(r.integers(0, max(s[-1], d[-1]))))
        while True:
            a, b = int(r.integers(0, 4)), int(r.integers(0, 4))
            O = (I[-1] - 1) * s[-1] - a - b + d[-1] * (k[-1] - 1) + op[-1] + 1
            if O >= 1:
                break
        pl.append(a)
        ph.append(b)
    x = r.standard_normal((B, g * Cig) + tuple(I))
    w = r.standard_normal((g * Cig, Cog) + tuple(k))
    bias = r.standard_normal(g * Cog) if r.random() < 0.7 else None
    return x, w, bias, s, pl, ph, d, op, g


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_matches_torch_conv_transpose_f64(nd):
    r = _rng(10 + nd)
    for _ in range(40):
        x, w, bias, s, pl, ph, d, op, g = _random_problem(r, nd)
        y = oracle.conv_transpose(x, w, bias, s, pl, ph, d, op, g)
        ref = _torch_convT(x, w, bias, s, pl, ph, d, op, g)
        assert y.shape == ref.shape
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# forward-convolution equivalence: dilate input by stride, reverse taps,
# pad d*(k-1) - pad_lo before and d*(k-1) - pad_hi + op after (crop if < 0)
# --------------------------------------------------------------------------

def _via_dilated_forward_conv(x, w, bias, s, pl, ph, d, op, g):
    nd = x.ndim - 2
    B, C_in = x.shape[:2]
    Cog = w.shape[1]
    k = w.shape[2:]
    # insert s-1 zeros between input samples on every axis
    shape = [B, C_in] + [(x.shape[2 + a] - 1) * s[a] + 1 for a in range(nd)]
    xd = np.zeros(shape)
    xd[(slice(None), slice(None)) + tuple(slice(None, None, s[a]) for a in range(nd))] = x
    # pad (or crop, where negative) each side: the padded sequence has length
    # L = n + lo + hi and its element j is the dilated input's element j - lo
    # (zero outside).  Padding both sides by P >= max(lo, hi, 0) and slicing
    # handles crops larger than the input too.
    for a in range(nd):
        lo = d[a] * (k[a] - 1) - pl[a]
        hi = d[a] * (k[a] - 1) - ph[a] + op[a]
        ax = 2 + a
        n = xd.shape[ax]
        L = n + lo + hi
        P = max(0, lo, hi)
        z = list(xd.shape); z[ax] = P
        big = np.concatenate([np.zeros(z), xd, np.zeros(z)], axis=ax)
        xd = np.take(big, range(P - lo, P - lo + L), axis=ax)
    # forward-conv weight [C_out, C_in/g, k...]: per group swap in/out, flip taps
    Cig = C_in // g
    blocks = []
    for gi in range(g):
        wg = w[gi * Cig:(gi + 1) * Cig]                 # [Cig, Cog, k...]
        wg = np.swapaxes(wg, 0, 1)                      # [Cog, Cig, k...]
        wg = np.flip(wg, axis=tuple(range(2, 2 + nd)))  # reversed taps
        blocks.append(wg)
    wf = np.ascontiguousarray(np.concatenate(blocks, axis=0))
    out = _CONV[nd](torch.from_numpy(np.ascontiguousarray(xd)), torch.from_numpy(wf),
                    None if bias is None else torch.from_numpy(bias),
                    stride=1, padding=0, dilation=tuple(d), groups=g).numpy()
    assert out.shape[1] == g * Cog
    return out


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_equals_forward_conv_of_dilated_input_with_flipped_kernel(nd):
    r = _rng(20 + nd)
    for _ in range(40):
        x, w, bias, s, pl, ph, d, op, g = _random_problem(r, nd)
        y = oracle.conv_transpose(x, w, bias, s, pl, ph, d, op, g)
        ref = _via_dilated_forward_conv(x, w, bias, s, pl, ph, d, op, g)
        assert y.shape == ref.shape
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# adjoint identity  <convT(x), y> = <x, conv(y)>
# --------------------------------------------------------------------------

def _conv_adjoint(yv, w, in_sp, s, pl, d, g):
    """conv(y)[b, ic, i] = sum_{oc in group, t} y[b, oc, i*s - pl + t*d] w[ic, oc_g, t].

    Written with torch's forward correlation: pad y by pl at the front and
    enough zeros at the back, convolve with stride s and dilation d, crop to I.
    """
    nd = yv.ndim - 2
    k = w.shape[2:]
    pads = []
    for a in reversed(range(nd)):
        need = (in_sp[a] - 1) * s[a] + d[a] * (k[a] - 1) + 1
        back = max(0, need - (yv.shape[2 + a] + pl[a]))
        pads += [pl[a], back]
    yp = F.pad(torch.from_numpy(yv), pads)
    out = _CONV[nd](yp, torch.from_numpy(w), None, stride=tuple(s), padding=0,
                    dilation=tuple(d), groups=g).numpy()
    sl = (slice(None), slice(None)) + tuple(slice(0, in_sp[a]) for a in range(nd))
    return out[sl]


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_adjoint_identity(nd):
    r = _rng(30 + nd)
    for _ in range(30):
        x, w, _, s, pl, ph, d, op, g = _random_problem(r, nd)
        y = oracle.conv_transpose(x, w, None, s, pl, ph, d, op, g)
        v = r.standard_normal(y.shape)
        lhs = float(np.sum(y * v))
        cv = _conv_adjoint(v, w, x.shape[2:], s, pl, d, g)
        assert cv.shape == x.shape
        rhs = float(np.sum(x * cv))
        scale = float(np.sum(np.abs(y * v))) + 1e-300
        assert abs(lhs - rhs) <= 1e-12 * scale


# --------------------------------------------------------------------------
# invariants and special cases
# --------------------------------------------------------------------------

def test_1x1_stride1_is_plain_gemm():
    r = _rng(40)
    x = r.standard_normal((3, 5, 4, 6))
    w = r.standard_normal((5, 7, 1, 1))
    bias = r.standard_normal(7)
    y = oracle.conv_transpose(x, w, bias)
    ref = np.einsum("io,bihw->bohw", w[:, :, 0, 0], x) + bias[None, :, None, None]
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_linearity_and_bias_shift():
    r = _rng(41)
    x1 = r.standard_normal((2, 4, 5, 3))
    x2 = r.standard_normal((2, 4, 5, 3))
    w = r.standard_normal((4, 3, 3, 2))
    bias = r.standard_normal(6)
    kw = dict(stride=(2, 3), pad_lo=(1, 0), pad_hi=(0, 1), dilation=(1, 2),
              output_padding=(1, 1), groups=2)
    y1 = oracle.conv_transpose(x1, w, None, **kw)
    y2 = oracle.conv_transpose(x2, w, None, **kw)
    y12 = oracle.conv_transpose(2.5 * x1 - 0.5 * x2, w, None, **kw)
    np.testing.assert_allclose(y12, 2.5 * y1 - 0.5 * y2, rtol=1e-12, atol=1e-12)
    yb = oracle.conv_transpose(x1, w, bias, **kw)
    np.testing.assert_allclose(yb - y1, np.broadcast_to(
        bias[None, :, None, None], y1.shape), rtol=0, atol=1e-12)


def test_empty_input_gives_bias_only():
    w = np.ones((0, 2, 3))
    x = np.ones((2, 0, 4))
    bias = np.array([0.5, -1.5])
    y = oracle.conv_transpose(x, w, bias, stride=(2,))
    assert y.shape == (2, 2, 9)
    np.testing.assert_array_equal(y, np.broadcast_to(bias[None, :, None], y.shape))
    x0 = np.ones((0, 3, 4))
    y0 = oracle.conv_transpose(x0, np.ones((3, 2, 3)), bias)
    assert y0.shape == (0, 2, 6)


def test_thread_count_does_not_change_bits():
    r = _rng(42)
    x, w, bias, s, pl, ph, d, op, g = _random_problem(r, 2)
    x = r.standard_normal((3,) + x.shape[1:])
    y1 = oracle.conv_transpose(x, w, bias, s, pl, ph, d, op, g, threads=1)
    y7 = oracle.conv_transpose(x, w, bias, s, pl, ph, d, op, g, threads=7)
    np.testing.assert_array_equal(y1, y7)


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_points_match_full_scatter(nd):
    r = _rng(50 + nd)
    for _ in range(25):
        x, w, bias, s, pl, ph, d, op, g = _random_problem(r, nd)
        y = oracle.conv_transpose(x, w, bias, s, pl, ph, d, op, g)
        idx = np.array(list(itertools.product(*[range(n) for n in y.shape])))
        v = oracle.points(x, w, bias, idx, s, pl, ph, d, op, g)
        np.testing.assert_array_equal(v, y.reshape(-1))


def test_low_precision_inputs_are_widened_exactly():
    x = torch.tensor([[[1.0 + 2 ** -7, -3.0]]], dtype=torch.bfloat16)
    w = torch.tensor([[[0.5, 2.0 ** -8]]], dtype=torch.float16)
    y = oracle.conv_transpose(x, w)
    a, b = 1.0 + 2 ** -7, -3.0
    p, q = 0.5, 2.0 ** -8
    np.testing.assert_array_equal(y[0, 0], [a * p, a * q + b * p, b * q])
