"""CPU oracle of the MoE layer forward pass (test infrastructure, not product code).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  It shares no code with the CUDA library.
"""

from .moe_oracle import (  # noqa: F401
    capacity,
    combine,
    expert_down,
    expert_down_fp8,
    expert_gate_up,
    expert_gate_up_fp8,
    gate_drop,
    grouped_ffn,
    moe_layer,
    moe_layer_tokens,
    permute,
    quantize_e4m3,
    quantize_rows_fp8,
    route,
    route_capacity,
    router_logits,
    silu,
    swiglu_ffn,
    topk_softmax,
)
