"""fp64 CPU oracle for the forward transposed convolution.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
CPU-baseline leg of the benchmark use it; the product never imports it.
"""
from .oracle import build, conv_transpose, out_shape, points, to_f64  # noqa: F401
