"""CPU oracle for the dense decoder forward pass (test infrastructure only).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark import
this package.  The product path never calls it and shares no code with it.
"""
from .model import (  # noqa: F401
    widen_bf16,
    round_bf16,
    rmsnorm,
    rope_rotate_half,
    rope_angles,
    gqa_attention,
    silu,
    linear,
    decode_step,
    prefill,
    causal_gqa_attention,
)
