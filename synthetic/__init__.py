"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA-side tests.

This package draws random numbers and lays them out; it computes nothing that the
MoE layer, the packer or the planner compute.  Both the oracle (``oracle/``) and the
product library are fed from here, so neither ever produces the other's inputs.
"""
from .gen import (  # noqa: F401
    LayerShape,
    SHAPES,
    block_id,
    block_shape,
    bf16_bits_from_f32,
    f32_from_bf16_bits,
    gen_block_np,
    gen_router_np,
    gen_shared_np,
    gen_token_np,
    gen_tokens_np,
    gen_phi_np,
    gen_q_assignment,
    gen_planner_offline_np,
    gen_kv_requests,
    zipf_log_prior,
    GATE_UP,
    DOWN,
)
