"""GB300-native conv2d input gradient (dgrad) as an implicit GEMM, with the
strided forward convolution, the fused RMSNorm + matmul and the attention
gradient with respect to V beside it.

The compute path is the C-ABI library ``libconv2d_grad_input.so`` built from
``csrc/`` for sm_103a; :mod:`.binding` marshals arguments to it.  Importing
this package does not load the library: the first call does, and it raises if
the library has not been built (there is no fallback path).
"""
from .binding import (  # noqa: F401
    DGRAD_BF16, DGRAD_DEBUG_SKIP_ARRIVE, DGRAD_F16, DGRAD_F32, DGRAD_KERNEL_AUTO,
    DGRAD_KERNEL_SIMT, DGRAD_KERNEL_TC, DGRAD_KERNEL_TC_POSM, DTYPE_CODE, PARAM_FIELDS, STATUS,
    DgradError, Params,
    conv2d_forward, conv2d_grad_input, conv2d_grad_input_check_errors, conv2d_grad_input_noalloc, conv2d_grad_input_pack_weight,
    conv2d_grad_input_prepacked, conv2d_grad_input_select_kernel, conv2d_grad_input_set_debug,
    conv2d_grad_input_set_kernel, conv2d_grad_input_set_wait_limit_ns,
    conv2d_grad_input_status_string, conv2d_grad_input_workspace_size, library, library_path,
    params_from_shapes,
    RmsParams, rmsnorm_matmul, rmsnorm_matmul_check_errors, rmsnorm_matmul_select_kernel,
    rmsnorm_matmul_set_kernel,
    MhaParams, mha_grad_v, mha_grad_v_check_errors, mha_grad_v_select_kernel, mha_grad_v_set_kernel,
)
