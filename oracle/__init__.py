"""fp64 CPU oracle for the shared-base, per-request LoRA projection (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
use this package. It shares no code with the CUDA path and imports nothing from it.
"""
from .lora_linear_oracle import (  # noqa: F401
    BM,
    bf16_bits_to_f64,
    check_segments,
    row_adapter_ids,
    lora_linear_fp64,
    lora_linear_merged_fp64,
    lora_linear_rows_fp64,
    merge_segments,
    plan_ref,
    max_rel_err,
    W4_GROUP,
    w4_dequantize_fp64,
    w4_weights_bf16_fp64,
    round_to_bf16_fp64,
    lora_linear_w4_fp64,
)
