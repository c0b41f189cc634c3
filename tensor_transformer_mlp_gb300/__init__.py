"""GB300-native tensor-parallel MLP block (Megatron TP/SP) behind the C ABI of libtpmlp.so.

The functions named tpmlp_* mirror the C entry points of include/tpmlp.h one to one;
``forward``, ``backward`` and ``sp_block`` allocate outputs with torch and call them.
The CUDA library is loaded on first use; there is no CPU fallback.
"""
from . import workloads  # noqa: F401
from ._binding import (  # noqa: F401
    SIGNATURES,
    TpmlpError,
    attention_backward,
    attention_forward,
    backward,
    forward,
    load_library,
    rmsnorm,
    rmsnorm_backward,
    sp_block,
    sp_block_backward,
    tpmlp_backward,
    tpmlp_backward_accumulate,
    tpmlp_backward_biased,
    tpmlp_backward_biased_workspace_size,
    tpmlp_backward_workspace_size,
    tpmlp_check_wait_timeout,
    tpmlp_device_status,
    tpmlp_forward,
    tpmlp_forward_biased,
    tpmlp_rmsnorm,
    tpmlp_rmsnorm_backward,
    tpmlp_rmsnorm_backward_workspace_size,
    tpmlp_set_gemm_variant,
    tpmlp_sp_block,
    tpmlp_sp_block_backward,
    tpmlp_sp_block_backward_workspace_size,
    tpmlp_sp_block_workspace_size,
    tpmlp_sp_dropout_grad_gather,
    tpmlp_sp_dropout_residual,
    tpmlp_sp_gather,
    tpmlp_sp_layernorm,
    tpmlp_sp_layernorm_backward,
    tpmlp_sp_layernorm_backward_workspace_size,
    tpmlp_sp_reduce_scatter,
)
