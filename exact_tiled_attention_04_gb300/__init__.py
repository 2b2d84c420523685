"""GB300-native fused exact attention (sm_103a): forward and backward.

O = softmax(scale * Q K^T) V and the per-row log-sum-exp, computed by fused
CUDA kernels that never write the N x N score matrix to HBM, and the
gradients dQ, dK, dV recomputed from the saved log-sum-exp.

The C ABI (include/fa.h) is mirrored one to one by ``binding``; ``inputs``
draws the seeded synthetic workloads.  Importing the package loads no CUDA
code; the first call into ``binding`` loads the library and fails loudly if it
was not built.
"""
from .binding import (FA_DTYPE_BF16, FA_DTYPE_F16, FA_DTYPE_F32, FA_FLAG_CAUSAL, FA_ERR_ALIGNMENT, FA_ERR_CUDA,  # noqa: F401
                      FA_ERR_INVALID_ARG, FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED, FA_OK, FAError,
                      attention, attention_backward, fa_bwd, fa_bwd_host, fa_bwd_host_workspace_size,
                      fa_bwd_validate, fa_bwd_workspace_size, fa_device_status, fa_fwd, fa_fwd_ex,
                      fa_fwd_ex_launches, fa_fwd_ex_splits, fa_fwd_ex_static, fa_fwd_ex_static_capacity, fa_fwd_ex_validate,
                      fa_fwd_ex_workspace_size, fa_fwd_host, fa_fwd_host_workspace_size, fa_fwd_validate,
                      fa_last_error_message, fa_selftest_barrier_timeout, fa_status_string,
                      fa_version)
