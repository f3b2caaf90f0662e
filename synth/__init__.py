"""Seeded synthetic inputs for the Gemma-4-E2B-shaped decoder: configs, weights, prompts.

This module is the synthetic stand-in for a checkpoint and a prompt set.  It is shared by the
CPU oracle (``oracle/``) and by the CUDA library's tests and benchmark, and it holds none of the
decoder's arithmetic: it only draws random numbers, rounds them to the storage formats a
checkpoint would use (bf16, packed int4 + bf16 group scales) and lays them out in the
canonical host format.

Shapes follow "Porting Gemma 4 E2B to SGLang-JAX on One Cloud TPU v5e", Step 1 (the E2B
config table: 35 layers, 20 KV-shared, per-layer input 256, one KV head, head_dim 256/512,
"4 sliding, 1 full, repeating") and Step 5 (double-wide MLP on the sharing layers, weight
names).  Widths the pages leave out (hidden 1536, 8 query heads, MLP 6144/12288, vocab
262144, window 512) are the synthetic workload's.

Canonical host int4 format ("Gemma 4 E2B in JAX on One TPU v5e", Step 3 and "One TPU chip,
eight agents", The engine: eight int4 values per int32, one bf16 scale per 32-element group):
element k of row n lives in word k // 8 of the row, bits [4*(k % 8), 4*(k % 8) + 4), as a
two's-complement nibble (low nibble first).  Scales are bf16 [N, K // 32].
"""
from .configs import CONFIGS, WORKLOADS, get_config, get_workload, layer_is_full, layer_mlp_width
from .weights import make_weights, make_model_weights, bf16_from_f32, linear_names, iter_linears, MODEL_DRAWS
from .prompts import make_prompts, replay_schedule

__all__ = [
    "CONFIGS", "WORKLOADS", "get_config", "get_workload", "layer_is_full", "layer_mlp_width",
    "make_weights", "make_model_weights", "MODEL_DRAWS", "bf16_from_f32", "linear_names", "iter_linears", "make_prompts",
    "replay_schedule",
]
