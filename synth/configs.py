"""Model shapes and workloads of the synthetic decoder.

Every field of a config is a plain number.  Fields the pages fix:
  num_layers, num_kv_shared_layers, ple_dim (hidden_size_per_layer_input), num_kv_heads,
  head_dim_sliding / head_dim_full, the "4 sliding, 1 full, repeating" layer pattern
  (full_every = 5) -- "Porting Gemma 4 E2B to SGLang-JAX on One Cloud TPU v5e", Step 1;
  mlp_shared = 2 * mlp on the sharing layers -- same page, Step 1 and Step 5;
  group_size 32 -- "Gemma 4 E2B in Pure JAX on a Colab TPU", introduction.
Fields the pages leave open carry the readings listed with each constant below.
"""
import copy

# Readings of constants the pages leave open (one value per config; both the oracle and the
# library receive them as inputs).
_OPEN = dict(
    rms_eps=1e-6,             # RMSNorm epsilon; the Rust rms_norm adds an unnamed eps
    rope_theta_sliding=10_000.0,
    rope_theta_full=1_000_000.0,
    attn_scale_sliding=0.0,   # 0 means 1/sqrt(head_dim)
    attn_scale_full=0.0,
    group_size=32,
    full_every=5,
    num_kv_heads=1,
)

CONFIGS = {
    # 5 layers (4 sliding window 64 then 1 full); last 2 KV-shared.
    "tiny": dict(_OPEN, name="tiny", num_layers=5, num_kv_shared_layers=2, hidden=256,
                 num_q_heads=4, head_dim_sliding=64, head_dim_full=128, sliding_window=64,
                 mlp=512, mlp_shared=1024, ple_dim=32, vocab=4096),
    # 10 layers, last 4 shared: exercises full-attention aliasing at tiny scale.
    "tiny10": dict(_OPEN, name="tiny10", num_layers=10, num_kv_shared_layers=4, hidden=256,
                   num_q_heads=4, head_dim_sliding=64, head_dim_full=128, sliding_window=64,
                   mlp=512, mlp_shared=1024, ple_dim=32, vocab=4096),
    # E2B head dims, window and MQA layout at a small width: long contexts in seconds.
    "mid": dict(_OPEN, name="mid", num_layers=10, num_kv_shared_layers=4, hidden=512,
                num_q_heads=8, head_dim_sliding=256, head_dim_full=512, sliding_window=512,
                mlp=1024, mlp_shared=2048, ple_dim=64, vocab=8192),
    # E2B-shaped.
    "e2b": dict(_OPEN, name="e2b", num_layers=35, num_kv_shared_layers=20, hidden=1536,
                num_q_heads=8, head_dim_sliding=256, head_dim_full=512, sliding_window=512,
                mlp=6144, mlp_shared=12288, ple_dim=256, vocab=262144),
}
# E2B layer shapes with an 8,192-entry vocabulary: every per-layer kernel is E2B's, while the
# whole model holds about 1 GB (small enough for multi-pass profiler captures).
CONFIGS["e2b-v8k"] = dict(CONFIGS["e2b"], name="e2b-v8k", vocab=8192)


def get_config(name):
    return copy.deepcopy(CONFIGS[name])


def layer_is_full(cfg, layer):
    """Layer pattern of the synthetic checkpoint: four sliding layers, then one full, repeating."""
    return layer % cfg["full_every"] == cfg["full_every"] - 1


def layer_mlp_width(cfg, layer):
    """MLP width stored for a layer: doubled from the first KV-shared index on."""
    first = cfg["num_layers"] - cfg["num_kv_shared_layers"]
    return cfg["mlp_shared"] if layer >= first else cfg["mlp"]


# Workloads: (config, weight format, batch, prompt length, output tokens).  "Output tokens"
# counts the token produced by the prefill, so a run makes out-1 decode steps.
WORKLOADS = {
    "tiny": dict(config="tiny", fmt="bf16", batch=1, prompt=16, out=16),
    "tiny-w4a16": dict(config="tiny", fmt="w4a16", batch=1, prompt=16, out=16),
    "tiny10": dict(config="tiny10", fmt="bf16", batch=1, prompt=16, out=16),
    "e2b-bf16-b1": dict(config="e2b", fmt="bf16", batch=1, prompt=128, out=512),
    "e2b-w4a16-b1": dict(config="e2b", fmt="w4a16", batch=1, prompt=128, out=512),
}
for _fmt in ("bf16", "w4a16"):
    for _b in (8, 16, 32, 64):
        WORKLOADS[f"e2b-{_fmt}-b{_b}"] = dict(config="e2b", fmt=_fmt, batch=_b, prompt=128,
                                               out=512)
WORKLOADS["e2b-v8k-w4a16-b1"] = dict(config="e2b-v8k", fmt="w4a16", batch=1, prompt=128, out=512)
WORKLOADS["e2b-v8k-w4a16-b64"] = dict(config="e2b-v8k", fmt="w4a16", batch=64, prompt=128, out=512)
# Agent replay: batch 8, 500-token start, 20 turns of 375 appended tokens + 32 outputs.
WORKLOADS["e2b-w4a16-replay-b8"] = dict(config="e2b", fmt="w4a16", batch=8, prompt=500,
                                        out=32, turns=20, turn_append=375)


def get_workload(name):
    w = copy.deepcopy(WORKLOADS[name])
    w["name"] = name
    return w
