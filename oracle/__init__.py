"""CPU fp64 oracle for the DeepSeekMoE layer forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import or run anything in this package.  The CUDA path
never does, and this package never imports the CUDA path: the two share no
code.  The one common dependency is ``moe_inputs`` (seeded random inputs,
no layer arithmetic).

See ``oracle/moe.py`` for the definitions and their sources,
``oracle/fp8.py`` for the e4m3 block-scaled expert FFN,
``oracle/backward.py`` for the gradients of the layer (Dgrad / Wgrad), and
``oracle/micro.py`` for the pure-Python scalar cross-check.
"""
from .moe import (  # noqa: F401
    sigmoid, silu, affinity, biased_topk, route, swiglu_ffn, permute,
    expert_ffn, combine, layer_forward, update_bias, relative_load,
    topk_near_tie_ok, group_limited_topk, group_topk_near_tie_ok,
)
