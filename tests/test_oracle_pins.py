"""Pins of the CPU oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a printed number, a
closed form, an invariant, a special case reducing to a textbook result, or brute force."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _pack_row(q):
    """Hand packing of one row of int4 values in the canonical layout (low nibble first)."""
    words = []
    for w in range(len(q) // 8):
        v = 0
        for j in range(8):
            v |= (int(q[8 * w + j]) & 0xF) << (4 * j)
        words.append(v)
    return np.array(words, dtype=np.uint32).view(np.int32)


def _bf16(x):
    return np.array([x], np.float32).view(np.uint32)[0] >> 16


# ---------------------------------------------------------------------------------- dequant
def test_dequant_levels_exact():
    # q = -8..7 twice, scale 0.5: every product is exactly representable.
    q = np.array(list(range(-8, 8)) * 2)
    packed = _pack_row(q)[None]
    scales = np.array([[_bf16(0.5)]], np.uint16)
    w = oracle.dequant_w4a16(packed, scales)
    np.testing.assert_array_equal(w[0], q * 0.5)


def test_dequant_nibble_order_probe():
    # One non-zero nibble at each position k: exactly element k is non-zero.
    for k in range(32):
        q = np.zeros(32, int)
        q[k] = 3
        w = oracle.dequant_w4a16(_pack_row(q)[None], np.array([[_bf16(1.0)]], np.uint16))
        assert np.nonzero(w[0])[0].tolist() == [k]
        assert w[0, k] == 3.0


def test_dequant_extreme_levels_and_group_scales():
    # Groups whose largest weight sits on level 7 or -8 (the QAT grid's two top levels),
    # each group with its own scale.
    q = np.array([7] * 32 + [-8] * 32)
    scales = np.array([[_bf16(0.25), _bf16(3.0)]], np.uint16)
    w = oracle.dequant_w4a16(_pack_row(q)[None], scales)
    assert np.all(w[0, :32] == 1.75) and np.all(w[0, 32:] == -24.0)


def test_dequant_rounds_to_bf16_nearest_even():
    # s = 1 + 1/128, q = 3: 3.0234375 lies exactly between bf16 3.015625 and 3.03125 -> even (3.03125)
    # s = 1 + 3/128, q = 3: 3.0703125 between 3.0625 and 3.078125 -> even (3.0625)
    # s = 1 + 1/128, q = 5: 5.0390625 -> below the midpoint -> 5.03125
    # s = 1 + 3/128, q = -3: symmetric -> -3.0625
    # s = 1 + 127/128, q = 7: 13.9453125, bf16 spacing 1/16 there -> 13.9375
    cases = [(3, 1 + 1 / 128, 3.03125), (3, 1 + 3 / 128, 3.0625), (5, 1 + 1 / 128, 5.03125),
             (-3, 1 + 3 / 128, -3.0625), (7, 1 + 127 / 128, 13.9375)]
    for q, s, want in cases:
        row = np.zeros(32, int)
        row[0] = q
        w = oracle.dequant_w4a16(_pack_row(row)[None], np.array([[_bf16(s)]], np.uint16))
        assert w[0, 0] == want, (q, s, w[0, 0], want)


def test_bf16_round_fp32_and_fp64_agree_on_exact_inputs():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(10000).astype(np.float32)
    a = oracle.bf16_round(x).astype(np.float64)
    b = oracle.bf16_round(x.astype(np.float64))
    np.testing.assert_array_equal(a, b)
    # Result is a bf16 value: low 16 bits zero; and the nearest one.
    bits = oracle.bf16_round(x).view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0)
    assert np.all(np.abs(oracle.bf16_round(x) - x) <= np.abs(x) * 2.0 ** -8)


# ---------------------------------------------------------------------------------- rmsnorm
def test_rmsnorm_constant_and_hand_case():
    g = np.array([1.0, 2.0, 0.5, -1.0], np.float64)
    out = oracle.rmsnorm(np.full(4, -3.0), g, 0.0)
    np.testing.assert_allclose(out, -g, rtol=1e-15)
    # [3, 4]: mean square 12.5
    out = oracle.rmsnorm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    np.testing.assert_allclose(out, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=1e-15)
    # eps enters under the square root: a zero vector stays zero, a tiny one is damped
    assert np.all(oracle.rmsnorm(np.zeros(8), np.ones(8), 1e-6) == 0)
    np.testing.assert_allclose(oracle.rmsnorm(np.full(2, 1e-3), np.ones(2), 1e-6),
                               1e-3 / math.sqrt(1e-6 + 1e-6), rtol=1e-12)


def test_rmsnorm_scale_invariance():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((3, 64))
    g = rng.standard_normal(64)
    np.testing.assert_allclose(oracle.rmsnorm(v * 37.5, g, 0.0), oracle.rmsnorm(v, g, 0.0),
                               rtol=1e-12)


# ------------------------------------------------------------------------------------- gelu
def test_gelu_tanh_identities():
    from scipy.special import erf
    z = np.linspace(-8, 8, 4001)
    g = oracle.gelu_tanh(z)
    # odd-part identity of x * Phi~(x) with Phi~(x) + Phi~(-x) = 1
    np.testing.assert_allclose(g - oracle.gelu_tanh(-z), z, atol=1e-12)
    # within the tanh form's known approximation error of the erf GELU
    exact = 0.5 * z * (1 + erf(z / math.sqrt(2)))
    assert np.max(np.abs(g - exact)) < 1e-3
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(oracle.gelu_tanh(np.array([20.0, -20.0])), [20.0, 0.0], atol=1e-12)


def test_gelu_tanh_against_logistic_closed_form():
    """The tanh form of GELU ("Porting Gemma 4 E2B to SGLang-JAX", Step 3: gelu with
    approximate=True) equals z * sigmoid(2u), u = sqrt(2/pi) (z + 0.044715 z^3), since
    (1 + tanh u) / 2 = 1 / (1 + exp(-2u)).  Written with exp instead of tanh, the points below
    pin the cubic term, its coefficient and the sqrt(2/pi) factor; the erf form of GELU differs
    from it by more than 1e-4 at z = 1, so an erf GELU in the oracle fails here."""
    def logistic_form(z):
        u = math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)
        return z / (1.0 + math.exp(-2.0 * u))

    points = [1.0, -0.5, 2.0, 0.25, -3.0]
    got = oracle.gelu_tanh(np.array(points, np.float64))
    for z, g in zip(points, got):
        assert abs(g - logistic_form(z)) <= 1e-12, (z, g)
    erf_gelu_1 = 0.5 * (1.0 + math.erf(1.0 / math.sqrt(2.0)))
    assert abs(got[0] - erf_gelu_1) > 1e-4
    # without the cubic term the value at z = 2 moves by ~2e-2
    u_lin = math.sqrt(2.0 / math.pi) * 2.0
    assert abs(got[2] - 2.0 / (1.0 + math.exp(-2.0 * u_lin))) > 1e-2


# ------------------------------------------------------------------------------------- rope
def test_rope_identity_norm_and_relative_position():
    d = 16
    cos, sin = oracle.rope_tables(10000.0, d, 64, np.float64)
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    np.testing.assert_allclose(oracle.apply_rope(q, cos[0], sin[0]), q, rtol=0, atol=0)
    for p in (1, 7, 63):
        r = oracle.apply_rope(q, cos[p], sin[p])
        h = d // 2
        np.testing.assert_allclose(r[:h] ** 2 + r[h:] ** 2, q[:h] ** 2 + q[h:] ** 2, rtol=1e-12)
    dots = [oracle.apply_rope(q, cos[m], sin[m]) @ oracle.apply_rope(k, cos[m - 5], sin[m - 5])
            for m in (5, 20, 40)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


def test_rope_is_complex_rotation():
    # Pair (i, i + d/2) of a unit vector rotates by angle p * theta^(-2i/d).
    d, theta = 8, 100.0
    cos, sin = oracle.rope_tables(theta, d, 10, np.float64)
    for i in range(d // 2):
        v = np.zeros(d)
        v[i] = 1.0
        r = oracle.apply_rope(v, cos[9], sin[9])
        ang = 9 * theta ** (-2.0 * i / d)
        assert abs(r[i] - math.cos(ang)) < 1e-12 and abs(r[i + d // 2] - math.sin(ang)) < 1e-12


# ---------------------------------------------------------------------------- masks / attend
@pytest.mark.parametrize("window", [1, 2, 3, 15, 16, 17])
def test_visible_keys_brute_force(window):
    T = 16
    for full in (False, True):
        dense = np.zeros((T, T), bool)
        for i in range(T):                      # brute force: every (query, key) pair
            for j in range(T):
                dense[i, j] = j <= i and (full or i - j < window)
        for p in range(T):
            got = np.zeros(T, bool)
            got[oracle.visible_keys(p, full, window)] = True
            assert np.array_equal(got, dense[p]), (p, full, window)


def test_attend_special_cases():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((4, 8))
    K = rng.standard_normal((1, 8))
    V = rng.standard_normal((1, 8))
    np.testing.assert_allclose(oracle.attend(q, K, V, 0.3), np.repeat(V, 4, 0), rtol=1e-15)
    K = rng.standard_normal((9, 8))
    V = rng.standard_normal((9, 8))
    np.testing.assert_allclose(oracle.attend(np.zeros((4, 8)), K, V, 1.0),
                               np.repeat(V.mean(0, keepdims=True), 4, 0), rtol=1e-13)
    # one dominant key
    K = np.zeros((5, 8))
    K[2, 0] = 1.0
    qq = np.zeros((1, 8))
    qq[0, 0] = 1e4
    np.testing.assert_allclose(oracle.attend(qq, K, V[:5], 1.0)[0], V[2], rtol=1e-12)


# ---------------------------------------------------------------------- schedule / sharing
def test_kv_share_map_e2b_literal():
    cfg = synth.get_config("e2b")
    want = list(range(15)) + [13, 13, 13, 13, 14] * 4
    assert oracle.kv_share_map(cfg) == want
    types = oracle.layer_types(cfg)
    assert [l for l, t in enumerate(types) if t == "full"] == [4, 9, 14, 19, 24, 29, 34]
    assert [oracle.mlp_width(cfg, l) for l in range(35)] == [6144] * 15 + [12288] * 20
    own = oracle.owns_kv(cfg)
    assert sum(own) == 15 and sum(o for o, t in zip(own, types) if t == "full") == 3


def test_kv_share_map_tiny_readings():
    assert oracle.kv_share_map(synth.get_config("tiny")) == [0, 1, 2, 2, 4]
    assert oracle.kv_share_map(synth.get_config("tiny10")) == [0, 1, 2, 3, 4, 5, 5, 5, 5, 4]


def test_printed_sizes_e2b():
    gold = json.load(open(os.path.join(GOLD, "e2b_printed_sizes.json")))
    cfg = synth.get_config("e2b")
    c = oracle.param_counts(cfg)
    assert c["n_linears"] == gold["packed_int4_linears"]["value"]
    # linears + embedding + table in bf16 fall short of the printed total by the norm gains
    short = gold["bf16_weight_bytes"]["value"] - c["bf16_bytes"]
    assert 0 <= short < 1_000_000, short
    assert round(c["w4a16_bytes"] / 1e9, 3) == gold["w4a16_weight_gb"]["value"]
    assert round(c["embed_bytes"] / 1e9, 3) == gold["lm_head_copy_gb"]["value"]
    assert round(c["ple_bytes"] / 1e9, 2) == gold["ple_table_gb"]["value"]
    assert oracle.kv_bytes_per_token(cfg) == gold["kv_bytes_per_token"]["value"]
    assert oracle.kv_bytes_per_token(cfg) // 2 == gold["kv_elements_per_token"]["value"]
    assert 256 * oracle.kv_bytes_per_token(cfg) == gold["cache_bytes_context_256"]["value"]
    assert oracle.kv_bytes_per_token(cfg, True) == gold["kv_cell_bytes_copy_every_layer"]["value"]
    assert sum(oracle.owns_kv(cfg)) == gold["kv_owning_layers"]["value"]
    assert round(8 * 8192 * oracle.kv_bytes_per_token(cfg) / 1e9, 2) == gold["kv_fleet_8x8192_gb"]["value"]


def test_printed_sizes_reject_plausible_mistakes():
    """The size pins fail for the nearby wrong schedules (a guard on the pins themselves)."""
    gold = json.load(open(os.path.join(GOLD, "e2b_printed_sizes.json")))
    cfg = synth.get_config("e2b")
    for k, v in (("mlp_shared", 6144), ("num_kv_shared_layers", 0), ("full_every", 4),
                 ("head_dim_full", 256)):
        bad = dict(cfg, **{k: v})
        c = oracle.param_counts(bad)
        ok = (c["n_linears"] == gold["packed_int4_linears"]["value"]
              and round(c["w4a16_bytes"] / 1e9, 3) == gold["w4a16_weight_gb"]["value"]
              and oracle.kv_bytes_per_token(bad) == gold["kv_bytes_per_token"]["value"])
        assert not ok, k


# ---------------------------------------------------------------------------------- int4 tables
def test_dequant_group_of_256_one_scale_per_layer_slice():
    # a per-layer-table row of two 256-wide layer slices, each with its own scale: the group
    # size comes from the scale count, so slice 1's scale must reach all of its 256 values
    q = np.array(list(range(-8, 8)) * 16 + [7, -8] * 128)
    scales = np.array([[_bf16(0.125), _bf16(2.0)]], np.uint16)
    w = oracle.dequant_w4a16(_pack_row(q)[None], scales)
    np.testing.assert_array_equal(w[0, :256], q[:256] * 0.125)
    np.testing.assert_array_equal(w[0, 256:], q[256:] * 2.0)


def test_int4_per_layer_table_bytes_match_printed_weight_tree():
    """Quantising the per-layer table to int4 took the measured weight tree from 6.618 to
    3.113 GB (One TPU chip, eight agents, Measured).  The saving (3.505 GB) is the bf16 table
    less half a byte per value and one bf16 scale per 256-wide layer slice; a scale per 32,
    64, 128 or 512 values, or no scale at all, misses the printed pair."""
    gold = json.load(open(os.path.join(GOLD, "e2b_printed_sizes.json")))
    before, after = gold["ple_int4_weight_tree_gb"]["value"]
    cfg = synth.get_config("e2b")
    V, n, P = cfg["vocab"], cfg["num_layers"] * cfg["ple_dim"], cfg["ple_dim"]
    bf16 = oracle.param_counts(cfg)["ple_bytes"]

    def saved(group):
        return (bf16 - oracle.int4_table_bytes(V, n, group)) / 1e9

    tol = 0.0011                                        # two figures printed to 3 decimals
    assert abs(saved(P) - (before - after)) <= tol
    for wrong in (32, 64, 128, 512):
        assert abs(saved(wrong) - (before - after)) > tol, wrong
    assert abs((bf16 - V * n // 2) / 1e9 - (before - after)) > tol


# ---------------------------------------------------------------------------------- int8 KV
def test_kv_int8_exact_rows_and_half_even_ties():
    s0 = np.float32(2.0 ** -5)
    c = np.array([127, -3, 0, 5, -127, 64, 1, -1], np.float32)
    codes, s = oracle.kv_int8_quantize(c * s0)
    assert s[0] == s0 and codes.dtype == np.int8
    assert codes.tolist() == c.astype(int).tolist()
    np.testing.assert_array_equal(oracle.kv_int8_dequantize(codes, s), c * s0)
    # v / s lands exactly on k + 1/2: round half to even
    v = np.array([127, 2.5, -2.5, 3.5, 0.5, -0.5, 1.5, -126.5], np.float32) * s0
    codes, s = oracle.kv_int8_quantize(v)
    assert s[0] == s0
    assert codes.tolist() == [127, 2, -2, 4, 0, 0, 2, -126]


def test_kv_int8_error_bound_absmax_and_sign():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal((64, 256)) * rng.uniform(0.01, 10.0, (64, 1))).astype(np.float32)
    codes, s = oracle.kv_int8_quantize(v)
    assert s.shape == (64, 1)
    vh = oracle.kv_int8_dequantize(codes, s, np.float64)
    # half a quantisation step, plus the fp32 roundings of v / s and c * s
    assert np.all(np.abs(vh - v.astype(np.float64)) <= s.astype(np.float64) * (0.5 + 3e-5))
    r = np.arange(64)
    j = np.argmax(np.abs(v), axis=-1)
    assert np.all(np.abs(codes[r, j].astype(int)) == 127)
    assert np.all(np.sign(codes[r, j]) == np.sign(v[r, j]))
    assert np.all(np.abs(codes.astype(int)) <= 127)
    # each row has its own scale: a row 1000x smaller still uses the full code range
    small = np.concatenate([v[:1], v[:1] * np.float32(1e-3)])
    c2, s2 = oracle.kv_int8_quantize(small)
    assert np.max(np.abs(c2[1].astype(int))) == 127 and np.array_equal(c2[0], c2[1])


def test_kv_int8_zero_row_and_power_of_two_scaling():
    codes, s = oracle.kv_int8_quantize(np.zeros((2, 16), np.float32))
    assert np.all(codes == 0) and np.all(s == 0)
    out = oracle.kv_int8_dequantize(codes, s)
    assert np.all(out == 0) and np.all(np.isfinite(out))
    v = np.random.default_rng(2).standard_normal((8, 64)).astype(np.float32)
    c1, s1 = oracle.kv_int8_quantize(v)
    c2, s2 = oracle.kv_int8_quantize(v * np.float32(8.0))
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s2, s1 * np.float32(8.0))


def test_kv_int8_bytes_per_token_and_printed_capacity():
    """int8 rows with one fp32 scale each take 9,336 B/token on E2B against 18,432 at bf16,
    1.974x.  The pages bisected the resident-token ceiling at context 8,192 at 1,425,408
    (bf16) and 2,818,048 (int8) tokens, 1.977x (Feasibility part 1), and report 1.82-1.98x
    capacity (Measured).  A bf16 scale per row would give 1.987x: outside both."""
    gold = json.load(open(os.path.join(GOLD, "e2b_printed_sizes.json")))
    cfg = synth.get_config("e2b")
    b16 = oracle.kv_bytes_per_token(cfg)
    b8 = oracle.kv_bytes_per_token(cfg, kv_dtype="int8")
    assert b16 == 18432 and b8 == 12 * 2 * (256 + 4) + 3 * 2 * (512 + 4) == 9336
    ceil = gold["kv_resident_tokens_ctx8192"]["value"]
    printed = ceil["int8"] / ceil["bf16"]
    lo, hi = gold["int8_kv_capacity_gain"]["value"]
    assert abs(b16 / b8 - printed) / printed < 3e-3
    assert lo <= b16 / b8 <= hi
    bf16_scale = b16 / (12 * 2 * (256 + 2) + 3 * 2 * (512 + 2))
    assert not (lo <= bf16_scale <= hi) and abs(bf16_scale - printed) / printed > 3e-3
