"""CPU oracle of the fused MoE layer -- test infrastructure only.

Imported by the tests, by the package smoke check, by the CPU-baseline leg
of the benchmark and by the report script numerics_delta.py; never by the
product path.  See moe_oracle.py.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (  # noqa: F401
    e4m3_decode, e4m3_encode_satfinite, dequant_fp8_block, dequant_int8_channel,
    quant_int8_per_row, max_padded, moe_align_block_size, fused_moe_fp8,
    fused_moe_int8, fused_moe_rows, silu, gate_softmax_topk, gate_grouped_sigmoid_topk,
    unpack_int4, dequant_int4_group, fused_moe_int4,
)
