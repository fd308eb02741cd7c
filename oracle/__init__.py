"""CPU oracle of the routed W4A16 MoE layer (test infrastructure only).

Only the tests, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` use this package; the CUDA library and its binding never do.
"""
from .moe_oracle import (  # noqa: F401
    GROUP,
    bf16_bits_to_f64,
    combine,
    dequant,
    expert_ffn,
    expert_ffn_rows,
    expert_matrices,
    fp16_bits_to_f32,
    layer_forward,
    layer_forward_tokens,
    pack_int4,
    permute,
    route_topk,
    silu,
    unpack_int4,
)
