"""Whole-decoder pins of the CPU oracle (CPU only, tiny shapes)."""
import numpy as np
import pytest

import oracle
import synth


@pytest.fixture(scope="module", params=["bf16", "w4a16"])
def tiny(request):
    cfg = synth.get_config("tiny10")
    w = synth.make_weights(cfg, request.param, seed=3, gain_std=0.1, layer_scale_std=0.1)
    return cfg, w


def test_weight_shapes_follow_oracle_schedule(tiny):
    cfg, w = tiny
    for l, lw in enumerate(w["layers"]):
        d = oracle.decoder.head_dim(cfg, l)
        assert lw["q"]["shape"] == (cfg["num_q_heads"] * d, cfg["hidden"])
        assert lw["gate"]["shape"] == (oracle.mlp_width(cfg, l), cfg["hidden"])


def test_cached_decode_matches_full_reforward(tiny):
    """Cached decode against re-running the whole sequence with dense masks (One TPU chip,
    eight agents, The engine).  fp64: agreement to roundoff.  fp32: the cache stores bf16,
    so fp32 noise can flip a K/V rounding; the bound covers those flips."""
    cfg, w = tiny
    pr = synth.make_prompts(cfg["vocab"], 1, 20, seed=5)
    for dtype, tol in ((np.float64, 1e-9), (np.float32, 1e-3)):
        o = oracle.Oracle(cfg, w, max_batch=1, max_context=96, dtype=dtype)
        r = o.generate(pr, 12, keep_logits=True)
        seq = np.concatenate([pr[0], r["tokens"][0, :-1]])
        full = o.forward_full(seq)
        assert np.max(np.abs(full[19:] - r["logits"][:, 0])) < tol
        # the window (64) binds only past 64 keys: also check a short window explicitly
    cfg2 = dict(cfg, sliding_window=3)
    o = oracle.Oracle(cfg2, w, max_batch=1, max_context=96, dtype=np.float64)
    r = o.generate(pr, 6, keep_logits=True)
    seq = np.concatenate([pr[0], r["tokens"][0, :-1]])
    assert np.max(np.abs(o.forward_full(seq)[19:] - r["logits"][:, 0])) < 1e-9


def test_shared_layers_read_exactly_their_source(tiny):
    cfg, w = tiny
    o = oracle.Oracle(cfg, w, max_batch=2, max_context=32, dtype=np.float64)
    rng = np.random.default_rng(0)
    for l in o.K:
        o.K[l][:] = oracle.bf16_round(rng.standard_normal(o.K[l].shape))
        o.Vc[l][:] = oracle.bf16_round(rng.standard_normal(o.Vc[l].shape))
    pos = np.array([20, 9])
    slots = np.array([1, 0])
    qs = {l: rng.standard_normal((2, cfg["num_q_heads"], oracle.decoder.head_dim(cfg, l)))
          for l in range(cfg["num_layers"])}
    base = {l: o.attention_layer(l, qs[l], slots, pos) for l in qs}
    for src in o.K:
        saved = o.K[src].copy()
        o.K[src][1, 18] += 0.5                       # a key every layer type can see at p=20
        for l in qs:
            moved = not np.array_equal(o.attention_layer(l, qs[l], slots, pos)[0], base[l][0])
            assert moved == (o.share[l] == src), (l, src)
            assert np.array_equal(o.attention_layer(l, qs[l], slots, pos)[1], base[l][1])
        o.K[src][:] = saved


def test_ple_with_zero_projection(tiny):
    cfg, w = tiny
    w0 = dict(w)
    pmp = w["ple_model_proj"]
    if "w" in pmp:
        w0["ple_model_proj"] = dict(pmp, w=np.zeros_like(pmp["w"]))
    else:
        w0["ple_model_proj"] = dict(pmp, scales=np.zeros_like(pmp["scales"]))
    o = oracle.Oracle(cfg, w0, max_batch=1, max_context=8, dtype=np.float64)
    toks = np.array([5, 4000, 17])
    _, ple = o.embed(toks)
    tab = oracle.bf16_bits_to_float(w["ple_table"][toks], np.float64).reshape(3, cfg["num_layers"], -1)
    np.testing.assert_allclose(ple, tab * np.sqrt(cfg["ple_dim"]) / np.sqrt(2.0), rtol=1e-15)


def test_ple_projection_chunks_have_unit_rms(tiny):
    cfg, w = tiny
    w0 = dict(w, ple_table=np.zeros_like(w["ple_table"]),
              ple_proj_norm=np.full(cfg["ple_dim"], 0x3F80, np.uint16))
    o = oracle.Oracle(dict(cfg, rms_eps=0.0), w0, max_batch=1, max_context=8, dtype=np.float64)
    _, ple = o.embed(np.array([1, 2, 3]))
    rms = np.sqrt(np.mean((ple * np.sqrt(2.0)) ** 2, axis=-1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-12)
    # with eps the chunk keeps its direction and shrinks
    o = oracle.Oracle(cfg, w0, max_batch=1, max_context=8, dtype=np.float64)
    _, ple_eps = o.embed(np.array([1, 2, 3]))
    cos = np.sum(ple * ple_eps, -1) / np.linalg.norm(ple, axis=-1) / np.linalg.norm(ple_eps, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-12)
    assert np.all(np.sqrt(np.mean((ple_eps * np.sqrt(2.0)) ** 2, axis=-1)) < 1.0)


def test_slots_and_batch_are_independent(tiny):
    cfg, w = tiny
    pr = synth.make_prompts(cfg["vocab"], 2, 10, seed=9)
    a = oracle.Oracle(cfg, w, max_batch=3, max_context=32, dtype=np.float64)
    ra = a.generate(pr, 5, slots=np.array([2, 0]))
    b = oracle.Oracle(cfg, w, max_batch=1, max_context=32, dtype=np.float64)
    for i in range(2):
        b.reset()
        rb = b.generate(pr[i:i + 1], 5)
        np.testing.assert_array_equal(rb["tokens"][0], ra["tokens"][i])
        np.testing.assert_allclose(rb["last_logits"][0], ra["last_logits"][i], rtol=0, atol=1e-12)


def test_fp32_tracks_fp64(tiny):
    cfg, w = tiny
    pr = synth.make_prompts(cfg["vocab"], 1, 16, seed=0)
    r32 = oracle.Oracle(cfg, w, 1, 48, np.float32).generate(pr, 8, keep_logits=True)
    r64 = oracle.Oracle(cfg, w, 1, 48, np.float64).generate(pr, 8, keep_logits=True)
    same = np.cumprod(r32["tokens"][0] == r64["tokens"][0]).sum()
    assert same >= 1
    assert np.max(np.abs(r32["logits"][:same] - r64["logits"][:same])) < 1e-3


def test_argmax_lowest_index_on_ties():
    x = np.array([[0.0, 3.0, 1.0, 3.0], [5.0, 5.0, 5.0, 5.0]])
    assert oracle.greedy_argmax(x).tolist() == [1, 0]


def _pack_int4(q):
    """[N, K] integers in [-8, 7] -> int32 [N, K/8], low nibble first (canonical layout)."""
    nib = (np.asarray(q).reshape(q.shape[0], -1, 8) & 0xF).astype(np.uint32)
    return np.bitwise_or.reduce(nib << (np.arange(8, dtype=np.uint32) * np.uint32(4)), axis=2).view(np.int32)


def test_int4_tables_holding_bf16_numbers_decode_as_those_bf16_tables():
    """Vocabulary tables in int4 (Six serving engines, Step 3; One TPU chip, eight agents,
    Measured): when every q * s is a bf16 number, the int4 tables must decode exactly as bf16
    tables holding those numbers -- the embedding gather, the per-layer rows and the tied
    lm_head all read the dequantised table, with the per-layer table's one scale per slice."""
    cfg = synth.get_config("tiny10")
    w = synth.make_weights(cfg, "w4a16", seed=3, gain_std=0.1, layer_scale_std=0.1)
    rng = np.random.default_rng(7)
    w4, wb = dict(w, tables="int4"), dict(w)
    V, H, P, L = cfg["vocab"], cfg["hidden"], cfg["ple_dim"], cfg["num_layers"]
    for name, cols, group in (("embed", H, 32), ("ple_table", L * P, P)):
        q = rng.integers(-8, 8, (V, cols))
        e = rng.integers(-9, -5, (V, cols // group)).astype(np.float64)
        s = np.exp2(e)                                   # powers of two: q * s is exact in bf16
        w4[name] = {"packed": _pack_int4(q), "scales": synth.bf16_from_f32(s.astype(np.float32)),
                    "shape": (V, cols)}
        wb[name] = synth.bf16_from_f32((q * np.repeat(s, group, axis=1)).astype(np.float32))
    pr = synth.make_prompts(V, 1, 12, seed=4)
    for kv in ("bf16", "int8"):
        ra = oracle.Oracle(cfg, w4, 1, 32, np.float64, kv_dtype=kv).generate(pr, 5, keep_logits=True)
        rb = oracle.Oracle(cfg, wb, 1, 32, np.float64, kv_dtype=kv).generate(pr, 5, keep_logits=True)
        np.testing.assert_array_equal(ra["logits"], rb["logits"])
        np.testing.assert_array_equal(ra["tokens"], rb["tokens"])
    # and the scale really is per slice: one slice's scale doubled moves only that layer's rows
    w4b = dict(w4, ple_table=dict(w4["ple_table"], scales=w4["ple_table"]["scales"].copy()))
    w4b["ple_table"]["scales"][:, 3] += np.uint16(0x80)  # bf16 exponent + 1: scale x 2
    o1 = oracle.Oracle(cfg, w4, 1, 8, np.float64)
    o2 = oracle.Oracle(cfg, w4b, 1, 8, np.float64)
    t1 = oracle.table_rows(o1.ple_table, np.array([9]), np.float64).reshape(L, P)
    t2 = oracle.table_rows(o2.ple_table, np.array([9]), np.float64).reshape(L, P)
    np.testing.assert_array_equal(t2[3], 2 * t1[3])
    np.testing.assert_array_equal(np.delete(t2, 3, 0), np.delete(t1, 3, 0))


def test_int8_kv_cache_rows_on_the_grid_and_full_reforward(tiny):
    """int8 K/V rows (One TPU chip, eight agents, Measured): every cached row lies on its own
    255-level grid (codes times max|row| / 127), and cached decode still equals the full
    re-forward that stores the same rows."""
    cfg, w = tiny
    pr = synth.make_prompts(cfg["vocab"], 1, 20, seed=5)
    o = oracle.Oracle(cfg, w, max_batch=1, max_context=96, dtype=np.float64, kv_dtype="int8")
    r = o.generate(pr, 10, keep_logits=True)
    seq = np.concatenate([pr[0], r["tokens"][0, :-1]])
    assert np.max(np.abs(o.forward_full(seq)[19:] - r["logits"][:, 0])) < 1e-9
    n = len(seq)
    for l in o.K:
        for C in (o.K[l], o.Vc[l]):
            rows = C[0, :n]
            s = np.max(np.abs(rows), axis=-1, keepdims=True) / 127.0
            c = rows / s
            assert np.max(np.abs(c - np.rint(c))) < 1e-4 and np.max(np.abs(c)) <= 127 + 1e-4
    # the bf16 cache is not on such a grid: the check tells the two apart
    ob = oracle.Oracle(cfg, w, max_batch=1, max_context=96, dtype=np.float64)
    ob.generate(pr, 2)
    rows = ob.K[0][0, :20]
    c = rows / (np.max(np.abs(rows), axis=-1, keepdims=True) / 127.0)
    assert np.max(np.abs(c - np.rint(c))) > 1e-2


def test_int8_kv_tracks_bf16_kv(tiny):
    """Teacher-forced: int8 rows move the logits by far less than their spread (the pages
    found int8 KV indistinguishable from bf16 in quality; this is only a sanity bound)."""
    cfg, w = tiny
    toks = synth.make_prompts(cfg["vocab"], 1, 24, seed=8)[0]
    a = oracle.Oracle(cfg, w, 1, 32, np.float64)
    b = oracle.Oracle(cfg, w, 1, 32, np.float64, kv_dtype="int8")
    for p, t in enumerate(toks):
        la = a.step([0], [t], [p])[0]
        lb = b.step([0], [t], [p])[0]
        cos = la @ lb / np.linalg.norm(la) / np.linalg.norm(lb)
        assert cos > 0.999, (p, cos)
