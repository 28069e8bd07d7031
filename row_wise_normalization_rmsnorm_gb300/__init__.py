"""GB300-native RMSNorm forward and backward (sm_103a CUDA kernels behind a C ABI).

The public functions take contiguous CUDA tensors (bf16, fp16 or fp32, rows of
length N on the last dimension; w and dw in the activations' type, or fp32
beside 16-bit activations) and launch on the current stream:

  rmsnorm_fwd(x, w)                       -> y, rstd
  rmsnorm_add_fwd(x, residual, w)         -> y, residual_out, rstd
  rmsnorm_fwd_fp8(x, w, scaling=...)      -> E4M3 y, rstd, scale_inv, amax
  layernorm_fwd(x, gamma, beta)           -> y, mean, rstd (dict)
  layernorm_bwd(dy, x, gamma, mean, rstd) -> dx, dgamma, dbeta (dict)
  rmsnorm_bwd(dy, x, w, rstd)             -> dx, dw
  rmsnorm_add_bwd(dy, dres, h, w, rstd)   -> dx (= dresidual), dw
  rmsnorm_bwd_workspace_bytes(M, N, dt)

The CUDA library is loaded on first use and must have been built
(``python -m row_wise_normalization_rmsnorm_gb300.build``); there is no CPU
fallback. ``inputs`` holds the seeded synthetic workloads.
"""
from ._binding import (  # noqa: F401
    OP_BWD,
    OP_FWD,
    OP_LN_BWD,
    RMSNORM_BF16,
    RMSNORM_F16,
    RMSNORM_F32,
    RMSNORM_OUT_BF16,
    RMSNORM_OUT_F16,
    RMSNORM_WEIGHT_F32,
    TORCH_DTYPE,
    LIB_PATH,
    Plan,
    RMSNormError,
    layernorm_bwd,
    layernorm_bwd_workspace_bytes,
    layernorm_fwd,
    lib,
    plan_query,
    rmsnorm_add_bwd,
    rmsnorm_add_fwd,
    rmsnorm_bwd,
    rmsnorm_bwd_ex,
    rmsnorm_bwd_workspace_bytes,
    rmsnorm_fwd,
    rmsnorm_fwd_ex,
    rmsnorm_fwd_fp8,
)
