"""GB300-native forward transposed convolution (ConvTranspose 1D/2D/3D).

The compute path is libct.so (hand-written CUDA for sm_103a behind the C ABI
in include/ct.h); this package is its thin ctypes binding.  Importing the
package does not load the library; the first call does, and raises if the
library has not been built.  There is no CPU fallback.
"""
from .ct import (  # noqa: F401
    CT_BF16, CT_F16, CT_F32, CT_OK, CT_ROUTE_AUTO, CT_ROUTE_BIAS_FILL, CT_ROUTE_GATHER,
    CT_ROUTE_GROUPED, CT_ROUTE_NONE, CT_ROUTE_SIMT_GEMM, CT_ROUTE_TC_GEMM,
    CT_ROUTE_TC32_GEMM, EXPORTS,
    ROUTE_NAMES, CtError, conv_transpose, ct_conv_transpose_nd, ct_conv_transpose_nd_host, ct_conv_transpose_nd_profiled,
    ct_conv_transpose_nd_noalloc, CT_NOALLOC_SCRATCH_BYTES,
    ct_conv_transpose_out_shape, ct_conv_transpose_route, ct_conv_transpose_kernel,
    ct_conv_transpose_workspace_bytes,
    ct_device_status, ct_host_buffers_release, ct_last_error, ct_status_string, ct_version,
    dtype_code, lib, ct_conv_transpose_backward_nd, ct_conv_transpose_backward_workspace_bytes,
    ct_conv_transpose_backward_kernels,
    conv_transpose_backward, ConvTransposeFunction, conv_transpose_autograd,
    ct_conv_transpose_nd_ex, ct_conv_transpose_ex_workspace_bytes, ACTIVATIONS, CT_ACT_NONE,
    CT_ACT_RELU, CT_ACT_LEAKY_RELU, CT_ACT_SILU, CT_ACT_GELU, CT_ACT_TANH, CT_ACT_SIGMOID,
    CT_W_TORCH, CT_W_KDHW_CI_CO, CT_W_KDHW_CO_CI, ct_set_wait_limit_ns,
    CT_WAIT_LIMIT_DEFAULT_NS)
