"""Plain CPU oracle of the Gemma-4-E2B-shaped greedy decoder (numpy; fp32, or fp64 as a
precision-ladder diagnostic).  TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check
and the benchmark's CPU-baseline leg; never by the CUDA library, with which it shares no code.

Sources (page title, section):
  [P1] "Gemma 4 E2B in JAX on One TPU v5e: bf16 or 4-Bit, Python or Rust, and How It Stands
       Against vLLM" -- Step 2 (jitted prefill, static KV cache, one decode step per token),
       Step 3 (W4A16 weights unpacked before every matmul), Step 4 (the Rust rms_norm).
  [P2] "Six serving engines on one Cloud TPU v5e chip (Gemma 4 E2B)" -- What Changes and
       What Stays, Step 3 (a build with the vocabulary tables and the lm_head in int4).
  [P3] "Porting Gemma 4 E2B to SGLang-JAX on One Cloud TPU v5e" -- Step 1 (config and layer
       pattern), Step 3 (per-layer embeddings: construction and per-layer mixing), Step 4 (a
       sharing layer applies RoPE to its queries only and reads its source's post-norm,
       post-RoPE K/V), Step 5 (double-wide MLP from the first sharing layer on).
  [P4] "Gemma 4 E2B in Pure JAX on a Colab TPU: Google's 4-Bit Export Against an Exact
       Repack" -- cell 2.2 (tied lm_head, 276 packed linears), cell 3.1 (int4 groups of 32).
  [P5] "One TPU chip, eight agents" -- The engine (kv_share_map, static cache, cached decode
       against a full re-forward, RoPE on logical position), Feasibility part 1 (18 KiB of KV
       per token; resident-token ceilings at bf16 and int8), Measured: the raw JAX decode
       kernel (int8 KV cache; the per-layer table in int4: weight tree 6.618 -> 3.113 GB),
       Two optimizations that didn't work (decode dequantises to bf16 and reads the full
       weight set per token).

What pins each part (tests/test_oracle_*.py):
  dequant_w4a16    hand-built groups with exact values, nibble-order probes, RNE ties,
                   groups of 256 (the per-layer table's one scale per layer slice)
  kv_int8_*        exact codes for rows on a power-of-two grid, half-even ties, the s/2
                   error bound, zero rows, power-of-two scale invariance; bytes per token
                   against the printed bf16 / int8 resident-token ceilings
  int4 tables      tables whose int4 values are exact bf16 numbers decode identically to
                   the bf16 tables; the per-layer table's bytes against the printed weight
                   tree before and after its int4 quantisation
  rmsnorm          constant vectors, scale invariance, a hand-computed case
  gelu_tanh        closed-form values (z * sigmoid(2u) at hand-picked points, which an erf
                   GELU or a dropped cubic term fails) and its distance to the erf GELU
  rope             identity at position 0, norm preservation, relative-position property
  visible_keys     brute-force dense masks for several windows
  attend           one key gives V_0; equal scores give the mean of V
  kv_share_map     the literal E2B map and the printed source rule
  param_counts     the printed weight totals (9.257 GB bf16, 6.559 GB W4A16, 276 packed
                   linears, 0.805 GB embedding, 4.70 GB per-layer table) and KV bytes per token
                   (18,432; 4,718,592 at context 256; 43,008 when every layer holds a copy)
  Oracle.step      cached decode against the full re-forward (forward_full); shared layers
                   move only when their source cache is perturbed; PLE with a zero projection
  Oracle (whole)   the constants the pages leave open (eps, RoPE theta, attention scale, norm
                   placement, gain form) are parity unpinned beyond self-consistency: no
                   trained weights or reference logits are available.
  GeGLU order      parity unpinned (self-consistency only): the pages print the activation of
                   the per-layer-input gate alone, so gelu on the MLP gate (not on up) is a
                   reading.
  embedding scale  parity unpinned (self-consistency only): x = E[t] * sqrt(H) parallels the
                   printed sqrt(P) of the per-layer table; the pages do not print it.
"""
import numpy as np

# ----------------------------------------------------------------------------------------
# bf16 and the W4A16 weight format
# ----------------------------------------------------------------------------------------


def bf16_bits_to_float(u16, dtype=np.float32):
    """bf16 bit patterns -> values (exact in fp32 and fp64)."""
    bits = np.asarray(u16).astype(np.uint32) << np.uint32(16)
    return bits.view(np.float32).astype(dtype, copy=False)


def bf16_round(x):
    """Round to the nearest bf16 value, ties to even; returns the same dtype as x.

    fp32: round the 32-bit pattern at bit 16.  fp64: round the 64-bit pattern at bit 45
    (bf16 keeps 8 significant bits), so fp64 values are not double-rounded through fp32."""
    x = np.asarray(x)
    if x.dtype == np.float32:
        b = x.view(np.uint32)
        r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
        return r.view(np.float32)
    if x.dtype == np.float64:
        b = x.view(np.uint64)
        half = np.uint64((1 << 44) - 1)
        r = (b + half + ((b >> np.uint64(45)) & np.uint64(1))) & ~np.uint64((1 << 45) - 1)
        return r.view(np.float64)
    raise TypeError(x.dtype)


def dequant_w4a16(packed, scales, dtype=np.float32):
    """W4A16 -> dense weights: W[n, k] = bf16(q[n, k] * s[n, k // G]).

    packed: int32 [N, K/8]; element k in word k // 8, bits 4*(k % 8).., two's complement.
    scales: bf16 bits [N, K/G]; the group size G = K / scales.shape[1] is 32 for the linears
    and the token embedding, ple_dim (one scale per layer slice; 256 in E2B) for the
    per-layer table.  The
    product q*s is exact (4-bit integer times an 8-bit significand); it is then rounded to
    bf16 as dequantising to bf16 does [P5, Two optimizations; P4, cell 1.2]."""
    packed = np.asarray(packed)
    n_out, words = packed.shape
    scales = np.asarray(scales)
    assert (words * 8) % scales.shape[1] == 0
    group = (words * 8) // scales.shape[1]
    u = packed.view(np.uint32)
    shifts = np.arange(8, dtype=np.uint32) * np.uint32(4)
    nib = (u[:, :, None] >> shifts) & np.uint32(0xF)
    q = nib.astype(np.int32).reshape(n_out, words * 8)
    q = np.where(q >= 8, q - 16, q)
    s = bf16_bits_to_float(scales, np.float64)
    s = np.repeat(s, group, axis=1)
    prod = q.astype(np.float64) * s                    # exact
    return bf16_round(prod).astype(dtype)


def table_rows(table, rows, dtype=np.float32):
    """Rows of a vocabulary table (token embedding or per-layer table): bf16 bits [V, n], or
    an int4 table {"packed", "scales"} dequantised row by row [P2, What Changes and What
    Stays, Step 3: int4 vocabulary tables and lm_head; P5, Measured: an int4 per-layer
    table]."""
    if isinstance(table, dict):
        return dequant_w4a16(table["packed"][rows], table["scales"][rows], dtype)
    return bf16_bits_to_float(table[rows], dtype)


# ----------------------------------------------------------------------------------------
# int8 KV rows
# ----------------------------------------------------------------------------------------


def kv_int8_quantize(v):
    """Symmetric int8 code of each K or V row (last axis) [P5, Measured: int8 KV cache].

    The pages give no granularity; the reading is one fp32 scale per stored row (one
    position of one layer's single KV head, K and V separately), taken in fp32:
      a = max_j |v_j|,  s = a / 127,  c_j = round_half_even(v_j / s) clipped to [-127, 127];
    an all-zero row has s = 0 and codes 0.  Returns (codes int8 [..., d], s fp32 [..., 1])."""
    v = np.asarray(v).astype(np.float32)
    a = np.max(np.abs(v), axis=-1, keepdims=True)
    s = a / np.float32(127.0)
    safe = np.where(s > 0, s, np.float32(1.0))
    c = np.rint(v / safe)
    c = np.where(s > 0, np.clip(c, -127, 127), 0)
    return c.astype(np.int8), s.astype(np.float32)


def kv_int8_dequantize(codes, s, dtype=np.float32):
    """Stored value of an int8 row: c_j * s, formed in fp32 (exact in fp64)."""
    return (codes.astype(np.float32) * s.astype(np.float32)).astype(dtype)


# ----------------------------------------------------------------------------------------
# Elementwise pieces
# ----------------------------------------------------------------------------------------


def rmsnorm(v, g, eps):
    """RMSNorm over the last axis: v / sqrt(mean(v^2) + eps) * g [P1, Step 4]."""
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + v.dtype.type(eps)) * g


def gelu_tanh(z):
    """GELU, tanh form (jax.nn.gelu approximate=True, [P3, Step 3])."""
    t = z.dtype.type
    c = t(np.sqrt(2.0 / np.pi))
    return t(0.5) * z * (t(1.0) + np.tanh(c * (z + t(0.044715) * z * z * z)))


def rope_tables(theta, d, n_pos, dtype=np.float32):
    """cos/sin [n_pos, d/2] for rotate-half RoPE: angle(p, i) = p * theta^(-2i/d), in fp64."""
    i = np.arange(d // 2, dtype=np.float64)
    inv = np.power(np.float64(theta), -2.0 * i / d)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def apply_rope(v, cos, sin):
    """Rotate-half RoPE on the last axis; pairs (i, i + d/2).  cos/sin broadcast to v[..., :d/2]."""
    h = v.shape[-1] // 2
    a, b = v[..., :h], v[..., h:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def greedy_argmax(logits):
    """Greedy next token: the lowest index among the maxima (np.argmax's rule)."""
    return np.argmax(logits, axis=-1)


# ----------------------------------------------------------------------------------------
# Layer schedule and KV sharing
# ----------------------------------------------------------------------------------------


def layer_types(cfg):
    """'4 sliding, 1 full, repeating' [P3, Step 1]: layer l is full iff l % 5 == 4."""
    e = cfg["full_every"]
    return ["full" if l % e == e - 1 else "sliding" for l in range(cfg["num_layers"])]


def kv_share_map(cfg):
    """Source layer of each layer's K/V [P5, The engine; P3, Step 1].

    first = L - n_shared; a layer below `first` is its own source; a layer at or above it
    reads the K/V of the last layer below `first` of its own type.  Where no layer below
    `first` has that type (the 5-layer tiny model's last, full layer), the layer computes
    and keeps its own K/V -- the printed map has no entry for that case."""
    types = layer_types(cfg)
    first = cfg["num_layers"] - cfg["num_kv_shared_layers"]
    last_of = {}
    for i in range(first):
        last_of[types[i]] = i
    return [i if i < first else last_of.get(types[i], i) for i in range(cfg["num_layers"])]


def owns_kv(cfg):
    return [src == l for l, src in enumerate(kv_share_map(cfg))]


def mlp_width(cfg, l):
    """MLP width 2x from the first KV-shared layer on [P3, Step 5]."""
    first = cfg["num_layers"] - cfg["num_kv_shared_layers"]
    return cfg["mlp_shared"] if l >= first else cfg["mlp"]


def head_dim(cfg, l):
    return cfg["head_dim_full"] if layer_types(cfg)[l] == "full" else cfg["head_dim_sliding"]


def visible_keys(p, full, window):
    """Keys a query at position p attends to: all j <= p (full), or the `window` most
    recent ones, p - window < j <= p (sliding)."""
    lo = 0 if full else max(0, p - window + 1)
    return np.arange(lo, p + 1)


def attend(q, K, V, scale):
    """Softmax attention of query heads q [nq, d] over keys K, V [T, d] (one KV head):
    s = scale * q.K_j; a = softmax_j(s) with the max subtracted; o = sum_j a_j V_j."""
    s = (q @ K.T) * scale
    s = s - np.max(s, axis=-1, keepdims=True)
    e = np.exp(s)
    a = e / np.sum(e, axis=-1, keepdims=True)
    return a @ V


# ----------------------------------------------------------------------------------------
# Sizes that the pages print
# ----------------------------------------------------------------------------------------


def _linear_list(cfg):
    L, H, P = cfg["num_layers"], cfg["hidden"], cfg["ple_dim"]
    own = owns_kv(cfg)
    out = [("ple_model_proj", L * P, H)]
    for l in range(L):
        d = head_dim(cfg, l)
        F = mlp_width(cfg, l)
        nq = cfg["num_q_heads"] * d
        out.append((f"{l}.q", nq, H))
        if own[l]:
            out += [(f"{l}.k", d, H), (f"{l}.v", d, H)]
        out += [(f"{l}.o", H, nq), (f"{l}.gate", F, H), (f"{l}.up", F, H), (f"{l}.down", H, F),
                (f"{l}.ple_gate", P, H), (f"{l}.ple_proj", H, P)]
    return out


def param_counts(cfg):
    """Parameter and byte totals of the linears, embedding and per-layer table.

    Norm gains are not counted (well under 1 MB)."""
    lin = _linear_list(cfg)
    n_lin = sum(n * k for _, n, k in lin)
    embed = cfg["vocab"] * cfg["hidden"]
    ple = cfg["vocab"] * cfg["num_layers"] * cfg["ple_dim"]
    g = cfg["group_size"]
    return dict(
        n_linears=len(lin), linear_params=n_lin, embed_params=embed, ple_params=ple,
        bf16_bytes=2 * (n_lin + embed + ple),
        w4a16_bytes=n_lin // 2 + 2 * (n_lin // g) + 2 * (embed + ple),
        embed_bytes=2 * embed, ple_bytes=2 * ple,
    )


def kv_bytes_per_token(cfg, copy_to_every_layer=False, kv_dtype="bf16"):
    """K+V bytes per token: one KV head per layer that keeps a cache; bf16 values, or int8
    codes plus one fp32 scale per row."""
    own = owns_kv(cfg)
    layers = range(cfg["num_layers"]) if copy_to_every_layer else [l for l in range(cfg["num_layers"]) if own[l]]
    if kv_dtype == "int8":
        return sum(2 * cfg["num_kv_heads"] * (head_dim(cfg, l) + 4) for l in layers)
    assert kv_dtype == "bf16"
    return sum(2 * 2 * cfg["num_kv_heads"] * head_dim(cfg, l) for l in layers)


def int4_table_bytes(n_rows, n_cols, group):
    """Bytes of a vocabulary table in int4: half a byte per value plus a bf16 scale per group."""
    return n_rows * n_cols // 2 + 2 * (n_rows * n_cols // group)


# ----------------------------------------------------------------------------------------
# The decoder
# ----------------------------------------------------------------------------------------


class Oracle:
    """Greedy decoder over a per-sequence static KV cache (bf16 or int8 K/V, one KV head).

    Per token id t at position p [P3, Steps 3-5; P5, The engine]:
      x = E[t] * sqrt(H)
      tok = T_ple[t] * sqrt(P); pr = RMSNorm((W_pmp x) * H^-1/2 per P-chunk); ple = (pr + tok) / sqrt 2
      per layer l: h = RMSNorm(x); q = RoPE(RMSNorm_head(W_q h)); K/V-owning layers store
        RoPE(RMSNorm_head(W_k h)) and W_v h at slot p, as bf16 or as int8 rows (kv_dtype);
        E and T_ple are bf16 tables or int4 tables dequantised on use; attention over the visible
        keys of the source layer's cache; x += RMSNorm(W_o o);
        m = RMSNorm(x); x += RMSNorm(W_d (gelu(W_g m) * (W_u m)));
        x += RMSNorm(W_pp (gelu(W_pg x) * ple_l)); x *= lambda_l
      logits = E RMSNorm(x) (tied lm_head [P4, cell 2.2]); next = argmax, lowest index on ties.
    """

    def __init__(self, cfg, weights, max_batch=1, max_context=None, dtype=np.float32,
                 workers=None, kv_dtype="bf16"):
        assert kv_dtype in ("bf16", "int8")
        self.kv_dtype = kv_dtype
        self.cfg = cfg
        self.dtype = dt = np.dtype(dtype)
        self.t = dt.type
        L, H, P = cfg["num_layers"], cfg["hidden"], cfg["ple_dim"]
        self.L, self.H, self.P, self.V = L, H, P, cfg["vocab"]
        self.types = layer_types(cfg)
        self.share = kv_share_map(cfg)
        self.own = owns_kv(cfg)
        self.eps = cfg["rms_eps"]
        self.max_batch = max_batch
        self.max_context = max_context or 4096
        self.fmt = weights["fmt"]

        def lin(x):
            if "w" in x:
                return bf16_bits_to_float(x["w"], dt)
            return dequant_w4a16(x["packed"], x["scales"], dt)

        def gain(u16):
            return bf16_bits_to_float(u16, dt)

        jobs = [("pmp", weights["ple_model_proj"])]
        for l, lw in enumerate(weights["layers"]):
            names = ["q", "o", "gate", "up", "down", "ple_gate", "ple_proj"]
            if self.own[l]:
                names += ["k", "v"]
            jobs += [((l, n), lw[n]) for n in names]
        from concurrent.futures import ThreadPoolExecutor
        import os
        nw = workers or max(1, len(os.sched_getaffinity(0)))
        with ThreadPoolExecutor(nw) as ex:
            mats = list(ex.map(lambda j: lin(j[1]), jobs))
        self.W = {k: m for (k, _), m in zip(jobs, mats)}
        self.E = table_rows(weights["embed"], slice(None), dt)   # also the tied lm_head
        self.ple_table = weights["ple_table"]            # bf16 bits or int4; rows gathered per token
        self.g_ppn = gain(weights["ple_proj_norm"])
        self.g_final = gain(weights["final_norm"])
        self.lw = []
        for l, lw in enumerate(weights["layers"]):
            self.lw.append({k: gain(lw[k]) for k in ("in_norm", "post_attn_norm", "pre_ffw_norm",
                                                      "post_ffw_norm", "post_ple_norm", "q_norm",
                                                      "k_norm")})
            self.lw[-1]["layer_scale"] = self.t(lw["layer_scale"])
        self.sqrt_h = self.t(np.sqrt(np.float64(H)))
        self.inv_sqrt_h = self.t(1.0 / np.sqrt(np.float64(H)))
        self.sqrt_p = self.t(np.sqrt(np.float64(P)))
        self.inv_sqrt2 = self.t(1.0 / np.sqrt(np.float64(2.0)))
        self.rope = {}
        self.scale = {}
        for typ in ("sliding", "full"):
            d = cfg["head_dim_full"] if typ == "full" else cfg["head_dim_sliding"]
            theta = cfg["rope_theta_full"] if typ == "full" else cfg["rope_theta_sliding"]
            self.rope[typ] = rope_tables(theta, d, self.max_context, dt)
            s = cfg["attn_scale_full"] if typ == "full" else cfg["attn_scale_sliding"]
            self.scale[typ] = self.t(s if s != 0.0 else 1.0 / np.sqrt(np.float64(d)))
        self.reset()

    # -- cache ------------------------------------------------------------------------------
    def reset(self):
        """Fresh cache: per owning layer K and V [max_batch, max_context, d] of stored values
        (bf16 numbers, or int8 codes times their row scale)."""
        self.K, self.Vc = {}, {}
        for l in range(self.L):
            if self.own[l]:
                d = head_dim(self.cfg, l)
                self.K[l] = np.zeros((self.max_batch, self.max_context, d), self.dtype)
                self.Vc[l] = np.zeros((self.max_batch, self.max_context, d), self.dtype)

    # -- pieces -----------------------------------------------------------------------------
    def embed(self, tokens):
        x = self.E[tokens] * self.sqrt_h
        tok = table_rows(self.ple_table, tokens, self.dtype) * self.sqrt_p
        tok = tok.reshape(len(tokens), self.L, self.P)
        pr = (x @ self.W["pmp"].T) * self.inv_sqrt_h
        pr = rmsnorm(pr.reshape(len(tokens), self.L, self.P), self.g_ppn, self.eps)
        ple = (pr + tok) * self.inv_sqrt2
        return x, ple

    def _qkv(self, l, h, positions):
        """Query heads (normed, RoPE'd) and, for owning layers, the new K and V rows."""
        cfg, t = self.cfg, self.types[l]
        d = head_dim(cfg, l)
        n = h.shape[0]
        g = self.lw[l]
        cos, sin = self.rope[t]
        cp, sp = cos[positions][:, None, :], sin[positions][:, None, :]
        q = (h @ self.W[(l, "q")].T).reshape(n, cfg["num_q_heads"], d)
        q = apply_rope(rmsnorm(q, g["q_norm"], self.eps), cp, sp)
        if not self.own[l]:
            return q, None, None
        k = (h @ self.W[(l, "k")].T).reshape(n, 1, d)
        k = apply_rope(rmsnorm(k, g["k_norm"], self.eps), cp, sp)[:, 0]
        v = h @ self.W[(l, "v")].T
        return q, self._stored(k), self._stored(v)

    def _stored(self, r):
        """The value a cache row holds: bf16(r), or its int8 code times its scale."""
        if self.kv_dtype == "int8":
            return kv_int8_dequantize(*kv_int8_quantize(r), dtype=self.dtype)
        return bf16_round(r)

    def _mlp_ple(self, l, x, ple_l):
        g = self.lw[l]
        m = rmsnorm(x, g["pre_ffw_norm"], self.eps)
        a = gelu_tanh(m @ self.W[(l, "gate")].T) * (m @ self.W[(l, "up")].T)
        x = x + rmsnorm(a @ self.W[(l, "down")].T, g["post_ffw_norm"], self.eps)
        pg = gelu_tanh(x @ self.W[(l, "ple_gate")].T) * ple_l
        x = x + rmsnorm(pg @ self.W[(l, "ple_proj")].T, g["post_ple_norm"], self.eps)
        return x * g["layer_scale"]

    def final_logits(self, x):
        return rmsnorm(x, self.g_final, self.eps) @ self.E.T

    def attention_layer(self, l, q, slots, positions):
        """Attention of layer l for query heads q [n, nq, d] over the cache of its source
        layer (itself, or the layer kv_share_map names)."""
        src = self.share[l]
        typ = self.types[l]
        o = np.empty_like(q)
        for i in range(q.shape[0]):
            j = visible_keys(int(positions[i]), typ == "full", self.cfg["sliding_window"])
            o[i] = attend(q[i], self.K[src][slots[i], j], self.Vc[src][slots[i], j],
                          self.scale[typ])
        return o

    # -- one decode step ----------------------------------------------------------------------
    def step(self, slots, tokens, positions, trace=None):
        """One token per sequence: tokens[i] at positions[i] of cache slot slots[i].
        Writes the owning layers' K/V at that position and returns logits [n, V].
        trace (optional dict) receives per layer the attention output and the residual
        stream after the layer: trace[("attn", l)], trace[("x", l)]."""
        slots = np.asarray(slots)
        tokens = np.asarray(tokens)
        positions = np.asarray(positions)
        assert np.all(positions < self.max_context) and np.all((tokens >= 0) & (tokens < self.V))
        x, ple = self.embed(tokens)
        for l in range(self.L):
            g = self.lw[l]
            typ = self.types[l]
            h = rmsnorm(x, g["in_norm"], self.eps)
            q, k, v = self._qkv(l, h, positions)
            if self.own[l]:
                self.K[l][slots, positions] = k
                self.Vc[l][slots, positions] = v
            o = self.attention_layer(l, q, slots, positions)
            if trace is not None:
                trace[("attn", l)] = o.reshape(len(tokens), -1).copy()
            x = x + rmsnorm(o.reshape(len(tokens), -1) @ self.W[(l, "o")].T, g["post_attn_norm"],
                            self.eps)
            x = self._mlp_ple(l, x, ple[:, l])
            if trace is not None:
                trace[("x", l)] = x.copy()
        return self.final_logits(x)

    # -- whole sequences ----------------------------------------------------------------------
    def prefill(self, slots, prompts, start_pos=None):
        """Teacher-forced steps over equal-length prompts [n, T]; returns the last logits."""
        prompts = np.asarray(prompts)
        n, T = prompts.shape
        start = np.zeros(n, np.int64) if start_pos is None else np.asarray(start_pos)
        logits = None
        for t in range(T):
            logits = self.step(slots, prompts[:, t], start + t)
        return logits

    def generate(self, prompts, n_out, slots=None, keep_logits=False):
        """Greedy decode: prefill the prompts, then n_out - 1 decode steps.

        Returns dict(tokens [n, n_out], last_logits [n, V], gaps [n_out, n] top-2 gaps,
        logits [n_out, n, V] if keep_logits)."""
        prompts = np.asarray(prompts)
        n, T = prompts.shape
        slots = np.arange(n) if slots is None else np.asarray(slots)
        logits = self.prefill(slots, prompts)
        toks, gaps, all_logits = [], [], []
        for s in range(n_out):
            nxt = greedy_argmax(logits)
            top2 = np.sort(logits, axis=-1)[:, -2:]
            gaps.append(top2[:, 1] - top2[:, 0])
            toks.append(nxt)
            if keep_logits:
                all_logits.append(logits.copy())
            if s + 1 < n_out:
                logits = self.step(slots, nxt, np.full(n, T + s))
        out = dict(tokens=np.stack(toks, 1).astype(np.int32), last_logits=logits,
                   gaps=np.stack(gaps))
        if keep_logits:
            out["logits"] = np.stack(all_logits)
        return out

    # -- the slow thing that obviously is: full re-forward, no cache ----------------------------
    def forward_full(self, tokens):
        """Logits at every position of one sequence, recomputed from scratch with dense
        causal / sliding-window masks and no cache [P5, The engine: cached decode against
        re-running the full model]."""
        tokens = np.asarray(tokens)
        T = len(tokens)
        pos = np.arange(T)
        x, ple = self.embed(tokens)
        kv = {}
        W = self.cfg["sliding_window"]
        for l in range(self.L):
            g = self.lw[l]
            typ = self.types[l]
            h = rmsnorm(x, g["in_norm"], self.eps)
            q, k, v = self._qkv(l, h, pos)
            if self.own[l]:
                kv[l] = (k, v)
            K, V = kv[self.share[l]]
            i, j = np.meshgrid(pos, pos, indexing="ij")
            mask = (j <= i) if typ == "full" else ((j <= i) & (j > i - W))
            s = np.einsum("thd,jd->thj", q, K) * self.scale[typ]
            s = np.where(mask[:, None, :], s, -np.inf)
            s = s - np.max(s, axis=-1, keepdims=True)
            e = np.exp(s)
            a = e / np.sum(e, axis=-1, keepdims=True)
            o = np.einsum("thj,jd->thd", a, V).reshape(T, -1)
            x = x + rmsnorm(o @ self.W[(l, "o")].T, g["post_attn_norm"], self.eps)
            x = self._mlp_ple(l, x, ple[:, l])
        return self.final_logits(x)
