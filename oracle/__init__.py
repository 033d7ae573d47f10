"""fp64 CPU oracle for the forward transposed convolution and its gradients.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
CPU-baseline leg of the benchmark use it; the product never imports it.
"""
from .oracle import (ACTIVATIONS, activation, build, conv_transpose,  # noqa: F401
                     conv_transpose_backward, out_shape, points, to_f64)
