"""Seeded synthetic weights in the canonical host format.

Draws (the synthetic workloads' recipe):
  * bf16 tensors (every linear of the bf16 model, the token embedding, the per-layer
    embedding table): N(0, std) drawn in fp32, rounded to bf16 round-to-nearest-even.
  * W4A16 linears: q ~ uniform integers in [-8, 7]; scale = bf16(|N(0, scale_std)|), one per
    32 input values; packed eight nibbles per int32, low nibble first.
  * int4 vocabulary tables (optional): drawn the same way, one scale per 32 values of an
    embedding row and one per 256-wide layer slice of a per-layer-table row.
  * RMSNorm gains: bf16(1 + N(0, gain_std)), i.e. exactly 1 at gain_std = 0; the query and
    key norms' gains are bf16(qk_gain * that) (qk_gain = 1 leaves them unchanged).
  * layer scales: 1 + N(0, layer_scale_std) in fp32 (exactly 1 at std 0).

Each tensor has its own stream, SeedSequence([seed, tensor id, chunk]), so tensors are
independent of the order in which they are drawn and large tensors fill in parallel.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import layer_is_full, layer_mlp_width

_CHUNK = 1 << 22
_LINEARS = ("q", "k", "v", "o", "gate", "up", "down", "ple_gate", "ple_proj")
_LAYER_NORMS = ("in_norm", "post_attn_norm", "pre_ffw_norm", "post_ffw_norm", "post_ple_norm")


def bf16_from_f32(a):
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    rounded = bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def _pool():
    return ThreadPoolExecutor(max(1, len(os.sched_getaffinity(0))))


def _chunked(n, seed, tid, fill, out, pool):
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, c])))
        out[lo:hi] = fill(rng, hi - lo)

    list(pool.map(work, range(nchunks)))


def _normal_bf16(shape, std, seed, tid, pool):
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)

    def fill(rng, m):
        a = rng.standard_normal(m, dtype=np.float32)
        a *= np.float32(std)
        return bf16_from_f32(a)

    _chunked(n, seed, tid, fill, out, pool)
    return out.reshape(shape)


def _gain_bf16(n, std, seed, tid, pool):
    if std == 0.0:
        return np.full(n, 0x3F80, np.uint16)          # bf16 1.0
    g = _normal_bf16((n,), std, seed, tid, pool).astype(np.uint32) << np.uint32(16)
    return bf16_from_f32(np.float32(1.0) + g.view(np.float32))


def _scaled_gain(g, factor):
    if factor == 1.0:
        return g
    return bf16_from_f32(np.float32(factor) * (g.astype(np.uint32) << np.uint32(16)).view(np.float32))


def _int4_linear(n_out, n_in, scale_std, seed, tid, pool, group=32):
    assert n_in % group == 0 and group % 8 == 0
    q = np.empty(n_out * n_in, np.int8)
    _chunked(q.size, seed, tid, lambda rng, m: rng.integers(-8, 8, m, dtype=np.int8), q, pool)
    nib = (q.reshape(n_out, n_in // 8, 8).astype(np.uint32) & np.uint32(0xF))
    shifts = (np.arange(8, dtype=np.uint32) * np.uint32(4))
    packed = np.bitwise_or.reduce(nib << shifts, axis=2).view(np.int32)
    s = np.empty(n_out * (n_in // group), np.uint16)

    def fill(rng, m):
        a = np.abs(rng.standard_normal(m, dtype=np.float32))
        a *= np.float32(scale_std)
        return bf16_from_f32(a)

    _chunked(s.size, seed, tid + 50_000, fill, s, pool)
    return {"packed": np.ascontiguousarray(packed), "scales": s.reshape(n_out, n_in // group),
            "shape": (n_out, n_in)}


def linear_names():
    return _LINEARS


def linear_shapes(cfg, layer):
    """(N, K) of every linear stored for a layer of the synthetic checkpoint."""
    H, P = cfg["hidden"], cfg["ple_dim"]
    d = cfg["head_dim_full"] if layer_is_full(cfg, layer) else cfg["head_dim_sliding"]
    F = layer_mlp_width(cfg, layer)
    nq = cfg["num_q_heads"] * d
    return {"q": (nq, H), "k": (d, H), "v": (d, H), "o": (H, nq), "gate": (F, H),
            "up": (F, H), "down": (H, F), "ple_gate": (P, H), "ple_proj": (H, P)}


def make_weights(cfg, fmt, seed=0, std=0.02, scale_std=0.004, gain_std=0.0,
                 layer_scale_std=0.0, embed_std=None, qk_gain=1.0, tables="bf16"):
    """Draw every tensor of the synthetic checkpoint.

    fmt: "bf16" (every linear bf16) or "w4a16" (linears int4 + bf16 group scales).
    tables: "bf16" (token embedding and per-layer-embedding table N(0, embed_std) in bf16) or
    "int4" (both drawn like the int4 linears: the embedding with a scale per 32 values, the
    per-layer table with one scale per 256-wide layer slice).  K and V projections are drawn for
    every layer, as a checkpoint that carries them everywhere would; a decoder reads those
    of the layers that compute their own K/V.  qk_gain < 1 softens the attention scores
    (they scale with qk_gain squared), which keeps deep random models well conditioned.
    """
    assert fmt in ("bf16", "w4a16") and tables in ("bf16", "int4")
    L, H, P, V = cfg["num_layers"], cfg["hidden"], cfg["ple_dim"], cfg["vocab"]
    estd = std if embed_std is None else embed_std
    with _pool() as pool:
        def linear(n_out, n_in, tid):
            if fmt == "bf16":
                return {"w": _normal_bf16((n_out, n_in), std, seed, tid, pool),
                        "shape": (n_out, n_in)}
            return _int4_linear(n_out, n_in, scale_std, seed, tid, pool)

        if tables == "bf16":
            embed = _normal_bf16((V, H), estd, seed, 1, pool)
            ple_table = _normal_bf16((V, L * P), estd, seed, 2, pool)
        else:
            embed = _int4_linear(V, H, scale_std, seed, 1, pool)
            ple_table = _int4_linear(V, L * P, scale_std, seed, 2, pool, group=P)
        w = {"fmt": fmt, "tables": tables,
             "embed": embed,
             "ple_table": ple_table,
             "ple_model_proj": linear(L * P, H, 3),
             "ple_proj_norm": _gain_bf16(P, gain_std, seed, 4, pool),
             "final_norm": _gain_bf16(H, gain_std, seed, 5, pool),
             "layers": []}
        for l in range(L):
            base = 1000 + 64 * l
            shapes = linear_shapes(cfg, l)
            lw = {}
            for i, name in enumerate(_LINEARS):
                lw[name] = linear(*shapes[name], base + i)
            for i, name in enumerate(_LAYER_NORMS):
                lw[name] = _gain_bf16(H, gain_std, seed, base + 20 + i, pool)
            d = shapes["k"][0]
            lw["q_norm"] = _scaled_gain(_gain_bf16(d, gain_std, seed, base + 30, pool), qk_gain)
            lw["k_norm"] = _scaled_gain(_gain_bf16(d, gain_std, seed, base + 31, pool), qk_gain)
            if layer_scale_std == 0.0:
                lw["layer_scale"] = 1.0
            else:
                rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, base + 40])))
                lw["layer_scale"] = float(np.float32(1.0 + layer_scale_std * rng.standard_normal()))
            w["layers"].append(lw)
    return w


# Draw parameters of each model as the workloads use it, beyond make_weights' defaults.  The
# E2B-shaped models draw their q/k-norm gains at 0.5: with unit gains this random 35-layer
# stack is chaotic after a few dozen tokens (attention scores reach |s| ~ 19 and the fp32
# decoder drifts from its fp64 twin by 2.6e-2 in the logits at 24 tokens), so no fp32
# implementation could be held to the logit tolerance; at 0.5 the scores shrink 4x and the
# fp32 / fp64 difference stays near 1e-6.  The pages give no norm gains for this shape.
MODEL_DRAWS = {"e2b": dict(qk_gain=0.5), "e2b-v8k": dict(qk_gain=0.5)}


def make_model_weights(cfg, fmt, seed=0, **overrides):
    """The weights a workload runs on: make_weights with the model's draw parameters
    (MODEL_DRAWS), which both the benchmark and the parity tests use."""
    kw = dict(MODEL_DRAWS.get(cfg["name"], {}))
    kw.update(overrides)
    return make_weights(cfg, fmt, seed=seed, **kw)


def iter_linears(weights):
    """(name, linear) for every linear tensor of a weight dict, in a fixed order."""
    yield "ple_model_proj", weights["ple_model_proj"]
    for l, lw in enumerate(weights["layers"]):
        for name in _LINEARS:
            yield f"layers.{l}.{name}", lw[name]
