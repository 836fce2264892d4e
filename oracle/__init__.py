"""fp64 CPU oracle of the deterministic MoE layer.

TEST INFRASTRUCTURE ONLY: ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only users.  The CUDA path never imports,
links or calls anything here, and nothing here imports the CUDA package.
"""
from .moe_ref import (  # noqa: F401
    NEAR_TIE, widen, bf16_round, silu, silu_grad, router_logits, routing_weights, route_ref,
    dispatch_ref,
    expert_ffn, moe_forward_ref, moe_backward_ref,
)
from .mx_ref import e4m3_round, mx_quantize, mx_fake  # noqa: F401
from .nvfp4_ref import e2m1_round, nvfp4_quantize, nvfp4_fake  # noqa: F401
