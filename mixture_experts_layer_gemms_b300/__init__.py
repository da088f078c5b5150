"""DeepSeekMoE layer forward, B300-native (sm_103a CUDA behind a C ABI).

Calls (same names as the C ABI without the ``moe_`` prefix): ``route``,
``permute``, ``expert_ffn``, ``combine``, ``update_bias``, plus
``pack_weights``, ``workspace_size``, ``get_device_error``,
``route_grouped`` and ``route_noalloc``.  ``MoELayer`` chains them for one forward.

The shared library is loaded on first use of any of these names; if
``libmoe_b300.so`` has not been built
(``python -m mixture_experts_layer_gemms_b300.build``) that use raises
ImportError -- there is no fallback.
"""
from importlib import import_module

_FROM_LIB = ("EXPORTED", "LIB", "LIB_PATH", "MOE_BF16", "MOE_F32", "MOE_FP8",
             "MoEError", "fp8_weight_bytes", "pack_weights_fp8",
             "x_perm_bytes",
             "MoeShape", "backward", "backward_workspace_size", "combine",
             "expert_ffn", "expert_ffn_part",
             "get_device_error",
             "last_launch_count", "make_shape", "pack_weights", "permute",
             "route", "route_grouped", "route_noalloc",
             "selftest_wait_timeout", "update_bias",
             "workspace_size")
_FROM_LAYER = ("Buffers", "MoELayer")

__all__ = list(_FROM_LIB + _FROM_LAYER)


def __getattr__(name):
    if name in _FROM_LIB:
        return getattr(import_module("._lib", __name__), name)
    if name in _FROM_LAYER:
        return getattr(import_module(".layer", __name__), name)
    raise AttributeError(name)
