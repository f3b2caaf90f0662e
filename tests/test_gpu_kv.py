"""KV-cache variants against the oracle, through the C ABI: int8 cache rows (one fp32 scale
per row) and the paged cache (page tables over a shared pool), alone and together.

The int8 rows follow "One TPU chip, eight agents", Measured: the raw JAX decode kernel (int8
KV cache); the oracle applies the same row code (oracle.kv_int8_quantize) to the same fp32
rows.  Paging ("Six serving engines on one Cloud TPU v5e chip", Step 3, page size 128) moves
no arithmetic: a paged run must give the static run's results, checked here against the
oracle with pages handed out out of order and reused after release.

Decoding is teacher-forced on the oracle's tokens, so every step's logits are compared; the
GPU's argmax must equal the oracle's wherever the oracle's top-2 gap exceeds GAP_TIE."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

LOGIT_TOL = 3e-2
GAP_TIE = 2e-3


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from accelerator_decode_gb300 import runtime
    return runtime


def forced(dec, prompts, ref, slots=None, paged=False, start=None):
    """Teacher-forced decode on the GPU: prefill, then feed the oracle's tokens.  Paged
    handles reserve each step's position first.  Returns argmaxes [n, n_out], logits
    [n_out, n, V]."""
    n = len(prompts)
    n_out = ref["tokens"].shape[1]
    slots = list(range(n)) if slots is None else list(slots)
    nxt, lg = dec.prefill(slots, prompts, start_pos=start, want_logits=True)
    torch.cuda.synchronize()
    toks, logits = [nxt.cpu().numpy().copy()], [lg.cpu().numpy().copy()]
    d_slots = torch.tensor(slots, dtype=torch.int32, device="cuda")
    p0 = [len(p) + (0 if start is None else start[i]) for i, p in enumerate(prompts)]
    pos = torch.tensor(p0, dtype=torch.int32, device="cuda")
    tok = torch.empty(n, dtype=torch.int32, device="cuda")
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    lgt = torch.empty(n, dec.cfg["vocab"], dtype=torch.float32, device="cuda")
    for s in range(1, n_out):
        if paged:
            for i, sl in enumerate(slots):
                dec.reserve(sl, p0[i] + s)
        tok.copy_(torch.from_numpy(np.asarray(ref["tokens"][:, s - 1], np.int32)).cuda())
        dec.decode_step(d_slots, tok, pos, out, lgt)
        torch.cuda.synchronize()
        toks.append(out.cpu().numpy().copy())
        logits.append(lgt.cpu().numpy().copy())
        pos += 1
    return np.stack(toks, 1), np.stack(logits)


def check(ref, toks, logits, label):
    err = float(np.max(np.abs(logits - ref["logits"])))
    assert err <= LOGIT_TOL, (label, err)
    ok = ref["gaps"].T > GAP_TIE
    assert np.all((toks == ref["tokens"]) | ~ok), label
    return err


@pytest.mark.parametrize("name,fmt", [("tiny", "bf16"), ("tiny10", "w4a16")])
def test_int8_kv_matches_oracle(rt, name, fmt):
    cfg = synth.get_config(name)
    w = synth.make_weights(cfg, fmt, seed=3, gain_std=0.1, layer_scale_std=0.05)
    prompts = synth.make_prompts(cfg["vocab"], 2, 14, seed=8)
    ref = oracle.Oracle(cfg, w, max_batch=2, max_context=64, kv_dtype="int8").generate(
        prompts, 18, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=2, max_context=64, kv_format="int8")
    toks, logits = forced(dec, list(prompts), ref)
    assert dec.device_error()[1] == 0
    dec.close()
    check(ref, toks, logits, f"int8 {name}/{fmt}")


def test_int8_kv_is_not_the_bf16_cache(rt):
    """The int8 run must follow the int8 oracle more closely than the bf16 one (it really
    stores codes), and its handle holds fewer bytes (the persistent step's buffers exist only
    for bf16 rows, so the difference is not the cache's alone)."""
    cfg = synth.get_config("tiny10")
    w = synth.make_weights(cfg, "bf16", seed=6)
    prompts = synth.make_prompts(cfg["vocab"], 1, 20, seed=2)
    r8 = oracle.Oracle(cfg, w, max_batch=1, max_context=64, kv_dtype="int8").generate(prompts, 10, keep_logits=True)
    r16 = oracle.Oracle(cfg, w, max_batch=1, max_context=64).generate(prompts, 10, keep_logits=True)
    d8 = rt.Decoder(cfg, w, max_batch=1, max_context=64, kv_format="int8")
    d16 = rt.Decoder(cfg, w, max_batch=1, max_context=64)
    _, lg8 = forced(d8, list(prompts), r8)
    e8 = np.max(np.abs(lg8 - r8["logits"]))
    e16 = np.max(np.abs(lg8 - r16["logits"]))
    assert e8 < e16, (e8, e16)
    own = [l for l in range(cfg["num_layers"]) if oracle.owns_kv(cfg)[l]]
    kv16 = sum(2 * 1 * 64 * oracle.decoder.head_dim(cfg, l) * 2 for l in own)
    kv8 = sum(2 * 1 * 64 * (oracle.decoder.head_dim(cfg, l) + 4) for l in own)
    assert d16.device_bytes() - d8.device_bytes() >= kv16 - kv8
    d8.close()
    d16.close()


def test_int8_kv_long_context_e2b_heads(rt):
    """E2B head dims (256 sliding / 512 full), window 512, 600-token prompt: several tiles
    per split, the window binding, and the merge."""
    cfg = synth.get_config("mid")
    w = synth.make_weights(cfg, "w4a16", seed=1, gain_std=0.1)
    prompts = synth.make_prompts(cfg["vocab"], 1, 600, seed=5)
    ref = oracle.Oracle(cfg, w, max_batch=1, max_context=640, kv_dtype="int8").generate(
        prompts, 6, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=1, max_context=640, kv_format="int8")
    toks, logits = forced(dec, list(prompts), ref)
    assert dec.device_error()[1] == 0
    dec.close()
    check(ref, toks, logits, "int8 mid 600")


@pytest.mark.parametrize("kv,mode", [("bf16", 0), ("bf16", 1), ("int8", 0)])
def test_paged_matches_oracle_out_of_order_pages(rt, kv, mode):
    """Pages of 16 positions, handed out interleaved between two sequences (neither holds a
    contiguous run of pool pages); mode 1 runs the persistent step (bf16 rows only)."""
    cfg = synth.get_config("tiny10")
    w = synth.make_weights(cfg, "w4a16", seed=9, gain_std=0.1)
    prompts = synth.make_prompts(cfg["vocab"], 2, 30, seed=12)
    ref = oracle.Oracle(cfg, w, max_batch=2, max_context=96, kv_dtype=kv).generate(prompts, 20, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=2, max_context=96, kv_format=kv, kv_page_size=16)
    if mode == 1:
        dec.set_step_mode(1)
    total = dec.pages_free()
    assert total == 2 * 6
    for n in range(16, 64, 16):             # interleave: slot 0 and slot 1 alternate pages
        dec.reserve(0, n)
        dec.reserve(1, n)
    toks, logits = forced(dec, list(prompts), ref, paged=True)
    assert dec.device_error()[1] == 0
    assert dec.pages_free() == total - 2 * 4  # 30 + 19 positions = 49 -> 4 pages each
    dec.close()
    check(ref, toks, logits, f"paged {kv} mode {mode}")


def test_paged_release_and_reuse(rt):
    """A released slot's pages go to the next sequence, which must see none of the old
    keys; the other sequence keeps decoding correctly throughout."""
    cfg = synth.get_config("tiny10")
    w = synth.make_weights(cfg, "bf16", seed=4, gain_std=0.1)
    pa = synth.make_prompts(cfg["vocab"], 1, 40, seed=21)
    pb = synth.make_prompts(cfg["vocab"], 1, 24, seed=22)
    pc = synth.make_prompts(cfg["vocab"], 1, 18, seed=23)
    dec = rt.Decoder(cfg, w, max_batch=2, max_context=64, kv_page_size=16, kv_pages=6)
    ra = oracle.Oracle(cfg, w, max_batch=1, max_context=64).generate(pa, 8, keep_logits=True)
    ta, la = forced(dec, list(pa), ra, slots=[0], paged=True)
    check(ra, ta, la, "paged seq a")
    assert dec.pages_free() == 6 - 3
    dec.release(0)
    assert dec.pages_free() == 6
    rb = oracle.Oracle(cfg, w, max_batch=1, max_context=64).generate(pb, 8, keep_logits=True)
    tb, lb = forced(dec, list(pb), rb, slots=[1], paged=True)
    check(rb, tb, lb, "paged seq b on a's pages")
    rc = oracle.Oracle(cfg, w, max_batch=1, max_context=64).generate(pc, 8, keep_logits=True)
    tc, lc = forced(dec, list(pc), rc, slots=[0], paged=True)
    check(rc, tc, lc, "paged seq c on the rest")
    assert dec.device_error()[1] == 0
    dec.close()


def test_paged_pool_limits(rt):
    """Reservation is all or nothing; a position without a page is reported by the device
    (its K/V row is not written) and the handle keeps working."""
    from accelerator_decode_gb300 import g4
    cfg = synth.get_config("tiny")
    w = synth.make_weights(cfg, "bf16", seed=1)
    dec = rt.Decoder(cfg, w, max_batch=2, max_context=64, kv_page_size=16, kv_pages=3)
    dec.reserve(0, 33)                               # 3 pages
    assert dec.pages_free() == 0
    with pytest.raises(g4.G4Error) as e:
        dec.reserve(1, 1)
    assert e.value.status == g4.G4_ERR_OOM
    with pytest.raises(g4.G4Error) as e:
        dec.reserve(1, 65)
    assert e.value.status == g4.G4_ERR_CONTEXT_OVERFLOW
    dec.release(0)
    prompts = synth.make_prompts(cfg["vocab"], 1, 8, seed=1)
    dec.prefill([1], list(prompts))                  # reserves positions 0..7 itself
    assert dec.pages_free() == 2
    slots = torch.tensor([1], dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    dec.decode_step(slots, tok, torch.tensor([20], dtype=torch.int32, device="cuda"), out)  # page 1 not held
    status, word = dec.device_error()
    assert word & g4.G4_DEV_BAD_POSITION
    dec.reserve(1, 9)
    dec.decode_step(slots, tok, torch.tensor([8], dtype=torch.int32, device="cuda"), out)
    assert dec.device_error()[1] == 0
    dec.close()


# ---------------------------------------------------------------------------------------------
# int4 vocabulary tables ("Six serving engines on one Cloud TPU v5e chip", What Changes and
# What Stays): the token embedding, the per-layer table and the tied lm_head in int4.
@pytest.mark.parametrize("name,fmt,batch", [("tiny", "bf16", 2), ("tiny10", "w4a16", 2), ("tiny10", "w4a16", 3),
                                            ("tiny10", "w4a16", 8)])
def test_int4_tables_match_oracle(rt, name, fmt, batch):
    """batch 8 puts the lm_head on the tensor-core GEMM; 2 and 3 on the staged kernel's argmax
    epilogue in decode steps (the GEMV in the prefill)."""
    cfg = synth.get_config(name)
    w = synth.make_weights(cfg, fmt, seed=13, gain_std=0.1, tables="int4")
    prompts = synth.make_prompts(cfg["vocab"], batch, 12, seed=30)
    ref = oracle.Oracle(cfg, w, max_batch=batch, max_context=64).generate(prompts, 14, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=batch, max_context=64)
    assert dec.table_format == "w4a16"
    toks, logits = forced(dec, list(prompts), ref)
    assert dec.device_error()[1] == 0
    dec.close()
    check(ref, toks, logits, f"int4 tables {name}/{fmt}/b{batch}")


def test_all_variants_together_e2b_heads(rt):
    """int4 tables, int8 cache rows and a paged cache at once, E2B head dims, 300 tokens."""
    cfg = synth.get_config("mid")
    w = synth.make_weights(cfg, "w4a16", seed=17, gain_std=0.1, tables="int4")
    prompts = synth.make_prompts(cfg["vocab"], 2, 300, seed=31)
    ref = oracle.Oracle(cfg, w, max_batch=2, max_context=384, kv_dtype="int8").generate(
        prompts, 6, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=2, max_context=384, kv_format="int8", kv_page_size=128)
    toks, logits = forced(dec, list(prompts), ref, paged=True)
    assert dec.device_error()[1] == 0
    dec.close()
    check(ref, toks, logits, "int4 tables + int8 paged")


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_mqa_attention_kernel_matches_oracle(rt, kv, monkeypatch):
    """The attention kernel that serves every query head of a sequence from one K/V tile
    load (used from 8 sequences on), forced on at batch 2: E2B head dims, 300-token prompts,
    several splits and tiles, the merge."""
    monkeypatch.setenv("G4_ATTN_MQA_MIN", "1")
    cfg = synth.get_config("mid")
    w = synth.make_weights(cfg, "w4a16", seed=27, gain_std=0.1)
    prompts = synth.make_prompts(cfg["vocab"], 2, 300, seed=41)
    ref = oracle.Oracle(cfg, w, max_batch=2, max_context=384, kv_dtype=kv).generate(prompts, 8, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=2, max_context=384, kv_format=kv)
    toks, logits = forced(dec, list(prompts), ref)
    assert dec.device_error()[1] == 0
    dec.close()
    check(ref, toks, logits, f"mqa {kv}")


def test_persistent_step_refuses_int8_rows_and_int4_tables(rt):
    """The persistent step reads bf16 cache rows and tables only: asking for it with int8 rows
    or int4 tables is refused on the host, and the default path keeps working."""
    from accelerator_decode_gb300 import g4
    cfg = synth.get_config("tiny")
    for kw, tables in (({"kv_format": "int8"}, "bf16"), ({}, "int4")):
        w = synth.make_weights(cfg, "bf16", seed=2, tables=tables)
        dec = rt.Decoder(cfg, w, max_batch=1, max_context=32, **kw)
        with pytest.raises(g4.G4Error) as e:
            dec.set_step_mode(1)
        assert e.value.status == g4.G4_ERR_UNSUPPORTED
        assert dec.step_mode(1) == 0
        prompts = synth.make_prompts(cfg["vocab"], 1, 8, seed=2)
        ref = oracle.Oracle(cfg, w, max_batch=1, max_context=32,
                            kv_dtype=kw.get("kv_format", "bf16")).generate(prompts, 4, keep_logits=True)
        toks, logits = forced(dec, list(prompts), ref)
        dec.close()
        check(ref, toks, logits, f"refused persistent step {kw} {tables}")
