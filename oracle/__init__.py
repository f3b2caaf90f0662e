"""CPU oracle of the Gemma-4-E2B-shaped greedy decode step -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this package.
The CUDA library never calls it, and it shares no code with the library: it is a plain numpy
restatement of the decoder the pages describe, slow and written to be checked by eye.

Parity status of each part (what pins it) is listed in ``oracle/decoder.py``.
"""
from .decoder import (
    Oracle, bf16_round, bf16_bits_to_float, dequant_w4a16, rmsnorm, gelu_tanh, rope_tables,
    apply_rope, layer_types, kv_share_map, owns_kv, mlp_width, visible_keys, attend,
    param_counts, kv_bytes_per_token, greedy_argmax, table_rows, kv_int8_quantize,
    kv_int8_dequantize, int4_table_bytes,
)

__all__ = [
    "Oracle", "bf16_round", "bf16_bits_to_float", "dequant_w4a16", "rmsnorm", "gelu_tanh",
    "rope_tables", "apply_rope", "layer_types", "kv_share_map", "owns_kv", "mlp_width",
    "visible_keys", "attend", "param_counts", "kv_bytes_per_token", "greedy_argmax",
    "table_rows", "kv_int8_quantize", "kv_int8_dequantize", "int4_table_bytes",
]
