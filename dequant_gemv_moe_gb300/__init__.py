"""Block-quantized GEMV and sparse-MoE kernels for one GB300 (sm_103a).

The compute runs in libdqmoe.so (hand-written CUDA behind a C ABI, see
include/dqmoe.h); this package is a thin torch-facing binding over it.
"""
from ._lib import BF16, F16, F32, Q4_K, Q6_K, Q8_0, DqError, MoeDesc, lib, status_string  # noqa: F401
from .ops import (ExpertCache, block_geometry, dequant, device_status, moe_forward,  # noqa: F401
                  moe_permute, moe_router, moe_workspace_size, qgemv, stage)
