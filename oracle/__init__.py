"""CPU oracle of the sparse int4 MoE block (test infrastructure only).

Imported by the test suite, the package smoke check and the benchmark's
CPU-baseline leg; never by the library.
"""
from .moe_oracle import (  # noqa: F401
    bf16_to_f64, dequantize, exact_logit, expert_matrices, expert_mlp, f64_to_bf16_bits, moe_block,
    moe_stack, permutation, residual_add, rms_norm, route, router_logits, select_topk, sigmoid,
    silu, softmax, unpack_int4,
)
