"""DeepSeekMoE layer forward, B300-native (sm_103a CUDA behind a C ABI).

Calls (same names as the C ABI without the ``moe_`` prefix): ``route``,
``permute``, ``expert_ffn``, ``combine``, ``update_bias``, plus
``pack_weights``, ``workspace_size`` and ``get_device_error``.  ``MoELayer``
chains them for one forward.  Importing fails if ``libmoe_b300.so`` has not
been built (``python -m mixture_experts_layer_gemms_b300.build``).
"""
from ._lib import (  # noqa: F401
    EXPORTED, LIB, LIB_PATH, MOE_BF16, MOE_F32, MoEError, MoeShape, combine,
    expert_ffn, get_device_error, last_launch_count, make_shape, pack_weights,
    permute, route, update_bias, workspace_size,
)
from .layer import Buffers, MoELayer  # noqa: F401
