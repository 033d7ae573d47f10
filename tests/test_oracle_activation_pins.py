"""Pins of the oracle's activation (applied after the convolution, the NKI
page's conv3d_transpose activation_fn), CPU only: values fixed by the
definitions, identities that tie the functions to one another, and float64
torch's own activations (library routines) on random inputs."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_values_fixed_by_the_definitions():
    a = oracle.activation
    assert a([-1.5, 0.0, 2.0], "relu").tolist() == [0.0, 0.0, 2.0]
    assert a([-2.0, 3.0], "leaky_relu", 0.1).tolist() == [-0.2, 3.0]
    assert a([0.0], "sigmoid").tolist() == [0.5]
    assert a([0.0], "tanh").tolist() == [0.0]
    assert a([0.0], "silu").tolist() == [0.0]
    assert a([0.0], "gelu").tolist() == [0.0]
    assert a([1.7, -0.3], "none").tolist() == [1.7, -0.3]
    # Phi(1) = (1 + erf(1/sqrt 2)) / 2 = 0.8413447460685429
    assert abs(a([1.0], "gelu")[0] - 0.8413447460685429) < 1e-15
    assert abs(a([1.0], "sigmoid")[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


def test_identities_between_the_functions():
    v = np.linspace(-6.0, 6.0, 241)
    a = oracle.activation
    # sigmoid(v) + sigmoid(-v) = 1; tanh(v) = 2 sigmoid(2v) - 1
    assert np.allclose(a(v, "sigmoid") + a(-v, "sigmoid"), 1.0, rtol=0, atol=1e-15)
    assert np.allclose(a(v, "tanh"), 2 * a(2 * v, "sigmoid") - 1, rtol=0, atol=1e-14)
    # silu(v) = v sigmoid(v), so silu(v) - silu(-v) = v; likewise gelu with Phi
    assert np.allclose(a(v, "silu"), v * a(v, "sigmoid"), rtol=0, atol=1e-14)
    assert np.allclose(a(v, "silu") - a(-v, "silu"), v, rtol=0, atol=1e-13)
    assert np.allclose(a(v, "gelu") - a(-v, "gelu"), v, rtol=0, atol=1e-13)
    # relu(v) - relu(-v) = v; leaky relu is v on the right, alpha v on the left
    assert np.array_equal(a(v, "relu") - a(-v, "relu"), v)
    assert np.allclose(a(v, "leaky_relu", 0.2), np.where(v >= 0, v, 0.2 * v), rtol=0, atol=0)


@pytest.mark.parametrize("name,fn", [
    ("relu", torch.nn.functional.relu),
    ("leaky_relu", lambda t: torch.nn.functional.leaky_relu(t, 0.05)),
    ("silu", torch.nn.functional.silu),
    ("gelu", torch.nn.functional.gelu),
    ("tanh", torch.tanh),
    ("sigmoid", torch.sigmoid),
])
def test_matches_torch_f64(name, fn):
    v = np.random.default_rng(5).standard_normal(4000) * 4
    got = oracle.activation(v, name, 0.05)
    ref = fn(torch.from_numpy(v)).numpy()
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)


def test_unknown_activation_is_rejected():
    with pytest.raises(ValueError):
        oracle.activation([1.0], 9)
