"""GB300 (sm_103a) routed-expert hot path: Python binding of the C ABI.

The compute happens in ``libmoe_gb300.so`` (hand-written CUDA, see ``csrc/``);
this module only marshals arguments through ctypes.  The entry points keep the
C names (``moe_plan_create``, ``moe_forward``, ...); ``MoePlan`` wraps them for
torch tensors (device memory and streams only).

There is no CPU path: importing works anywhere, but every compute call needs the
built library and a CUDA device and raises otherwise.
"""

from .binding import (  # noqa: F401
    MOE_BUF,
    MOE_ERR_BAD_IDS,
    MOE_ERR_CUDA,
    MOE_ERR_INVALID_ARG,
    MOE_ERR_STATE,
    MOE_ERR_TIMEOUT,
    MOE_ERR_UNSUPPORTED,
    MOE_ERR_WORKSPACE,
    MOE_OK,
    MOE_PREC_BF16,
    MOE_PREC_MXFP8,
    MOE_PREC_NVFP4,
    MOE_WS_HOST_STAGING,
    MOE_WS_TRAINING,
    MoeError,
    MoePlan,
    amax_bf16,
    gemm_bf16,
    lib,
    prepare_weights_mxfp8,
    prepare_weights_mxfp8_backward,
    prepare_weights_nvfp4,
    quantize_mxfp8,
)
